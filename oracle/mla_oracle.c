/*
 * mla_oracle.c -- plain, slow, fp64 CPU oracle for weight-absorbed MLA decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library under mla_latent_kv_71_b300/csrc.
 *
 * Every floating-point intermediate is an IEEE double.  Inputs may be given
 * as fp64, fp32 or bf16 bit patterns; they are widened exactly to double on
 * read and nothing is ever rounded back.
 *
 * Sources (five web pages on Multi-head Latent Attention), cited below as:
 *   [Mishra]  "Multi-head Latent Attention", Neel Mishra (neelmishra.github.io)
 *   [Zhang]   "Multi-Head Latent Attention" post, zhangchitc.github.io
 *   [llms]    "Multi-Head Latent Attention: How Low-Rank KV Compression
 *              Scales LLM Serving" (llms.blog)
 *
 * Notation: b sequence, t query token of the step, i head, j cached position;
 * d_c latent width, d_r decoupled-RoPE width, d_h per-head content width.
 * The cache row of position j is [c_j ; k^R_j] (d_c + d_r numbers).
 *
 * Readings where the pages are silent (the same list is kept in the design
 * notes): the score scale is passed in (the pages give 1/sqrt(d_h + d_r));
 * RoPE pairs (x_2k, x_2k+1) with angle pos * base^(-2k/d_r); LSE is the
 * natural log of the sum of exp(scaled score); a causal query t of a step
 * with T tokens sits at position len - T + t and sees positions 0..len-T+t;
 * a sequence that sees no position gets o = 0 and lse = -inf.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- input */

enum { ORC_F64 = 0, ORC_F32 = 1, ORC_BF16 = 2 };

/* Exact widening of one stored element to double. */
static double rd(const void* p, int dtype, int64_t idx) {
    if (dtype == ORC_F64) return ((const double*)p)[idx];
    if (dtype == ORC_F32) return (double)((const float*)p)[idx];
    /* bf16: the upper 16 bits of an IEEE binary32 */
    uint32_t bits = (uint32_t)((const uint16_t*)p)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ------------------------------------------------- cache-size accounting */

/*
 * Numbers cached per token per layer for each scheme.
 *   MHA: 2 h d_h                 [Mishra] "Step 1: a low-rank latent";
 *                                [Zhang] "Multi-head attention: every head
 *                                caches its own keys and values"
 *   GQA: 2 h_kv d_h, MQA: 2 d_h  [Mishra] "The full accounting" table
 *   MLA latent only: d_c         [Zhang] "Low-rank joint compression"
 *   MLA with decoupled RoPE: d_c + d_r
 *                                [Mishra] "Step 4: decoupled RoPE";
 *                                [llms] "Quantitative Comparison and
 *                                Serving Economics"
 * out[0..4] = {MHA, GQA, MQA, MLA latent only, MLA with RoPE key}.
 */
void orc_cache_numbers(int64_t h, int64_t d_h, int64_t h_kv, int64_t d_c,
                       int64_t d_r, int64_t* out) {
    out[0] = 2 * h * d_h;
    out[1] = 2 * h_kv * d_h;
    out[2] = 2 * d_h;
    out[3] = d_c;
    out[4] = d_c + d_r;
}

/*
 * Multiply-add counts for the content scores of one query against n cached
 * tokens, in the two orders of [Zhang] "Matrix absorption: compression that
 * also saves compute":
 *   key side   : every token expands k_j = W^UK c_j (hd x d_c), then q.k_j (hd)
 *   query side : q^T W^UK once (hd x d_c), then q_lat . c_j (d_c) per token
 * out[0] = key-side count, out[1] = query-side count.
 */
void orc_score_cost(int64_t n, int64_t hd, int64_t d_c, int64_t* out) {
    out[0] = n * (hd * d_c + hd);
    out[1] = hd * d_c + n * d_c;
}

/* ----------------------------------------------------------------- RoPE */

/*
 * Rotary embedding of one d_r-vector at position pos, in place.
 * The pages fix only that RoPE rotates by a position-dependent angle
 * ([Mishra] "Step 3: RoPE breaks it"; [llms] "The Positional Problem and
 * Decoupled RoPE"); the pairing and frequencies are the reading above.
 */
void orc_rope(double* x, int d_r, double pos, double base) {
    for (int k = 0; k < d_r / 2; ++k) {
        double theta = pow(base, -2.0 * k / (double)d_r);
        double ang = pos * theta;
        double cs = cos(ang), sn = sin(ang);
        double a = x[2 * k], b = x[2 * k + 1];
        x[2 * k] = a * cs - b * sn;
        x[2 * k + 1] = a * sn + b * cs;
    }
}

/* ------------------------------------------- absorbed route, per stage */

/*
 * Query-side absorption: q_lat[r,i,:] = W^UK_i^T q_nope[r,i,:].
 * W^UK is [H*d_h x d_c] with head i owning rows i*d_h .. (i+1)*d_h-1
 * ([llms] "Low-Rank Key-Value Joint Compression"), i.e. [H, d_h, d_c].
 * [llms] "Query Key Absorption"; [Mishra] "Step 2: absorb the up-projections".
 * q_nope [R,H,d_h] (dtype dq), w_uk [H,d_h,d_c] (dtype dw) -> q_lat [R,H,d_c].
 */
void orc_absorb_q(const void* q_nope, int dq, const void* w_uk, int dw,
                  int R, int H, int d_h, int d_c, double* q_lat) {
    #pragma omp parallel for collapse(2) schedule(static)
    for (int r = 0; r < R; ++r)
        for (int i = 0; i < H; ++i) {
            double* dst = q_lat + ((int64_t)r * H + i) * d_c;
            for (int c = 0; c < d_c; ++c) dst[c] = 0.0;
            for (int e = 0; e < d_h; ++e) {
                double qv = rd(q_nope, dq, ((int64_t)r * H + i) * d_h + e);
                int64_t wrow = ((int64_t)i * d_h + e) * d_c;
                for (int c = 0; c < d_c; ++c) dst[c] += qv * rd(w_uk, dw, wrow + c);
            }
        }
}

/* Number of cached positions query t of sequence b sees. */
static int64_t visible_len(int64_t len, int T, int t, int causal) {
    int64_t n = causal ? len - (T - 1 - t) : len;
    return n < 0 ? 0 : n;
}

/*
 * Absorbed decode attention against the paged latent cache, for one
 * (b, t, i):
 *   s_j  = (q_lat . c_j + q_pe . k^R_j) * scale
 *          ([llms] "Query Key Absorption": the absorbed content score plus
 *          the decoupled RoPE score; [Zhang] "Value absorption": the sum is
 *          divided by sqrt(d_h + d_r) before the softmax)
 *   a_j  = softmax_j(s)  (two passes: maximum, then normalised exponentials)
 *   o    = sum_j a_j c_j ([llms] "Value Output Absorption": the weighted sum
 *          runs over the latents; W^UV is applied afterwards)
 *   lse  = m + ln sum_j exp(s_j - m)
 * Cache position j of sequence b lives in pool page page_table[b][j / page]
 * at row j % page; the pool row is [c (d_c) ; k^R (d_r)].
 * If a_out is not NULL it receives the n weights a_j.
 */
static void decode_one(const void* q_lat, int dql, const void* q_pe, int dqp,
                       const void* pool, int dp, const int32_t* page_table,
                       int64_t n, int b, int t, int i, int T, int H, int d_c,
                       int d_r, int page, int max_pages, double scale,
                       double* s /* scratch [n] */, double* o_row,
                       double* lse_out, double* a_out) {
    int64_t qrow = (((int64_t)b * T + t) * H + i);
    int64_t width = (int64_t)d_c + d_r;
    for (int c = 0; c < d_c; ++c) o_row[c] = 0.0;
    if (n == 0) {
        *lse_out = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        int64_t pg = page_table[(int64_t)b * max_pages + j / page];
        int64_t row = (pg * page + j % page) * width;
        double acc = 0.0;
        for (int c = 0; c < d_c; ++c)
            acc += rd(q_lat, dql, qrow * d_c + c) * rd(pool, dp, row + c);
        for (int e = 0; e < d_r; ++e)
            acc += rd(q_pe, dqp, qrow * d_r + e) * rd(pool, dp, row + d_c + e);
        s[j] = acc * scale;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) l += exp(s[j] - m);
    for (int64_t j = 0; j < n; ++j) {
        double a = exp(s[j] - m) / l;
        if (a_out) a_out[j] = a;
        int64_t pg = page_table[(int64_t)b * max_pages + j / page];
        int64_t row = (pg * page + j % page) * width;
        for (int c = 0; c < d_c; ++c) o_row[c] += a * rd(pool, dp, row + c);
    }
    *lse_out = m + log(l);
}

/*
 * Paged absorbed decode for every (b, t, i), or only for the n_sel flattened
 * indices ((b*T + t)*H + i) listed in sel (sel == NULL: all of them).
 * q_lat [B,T,H,d_c], q_pe [B,T,H,d_r], pool [P,page,d_c+d_r],
 * page_table [B,max_pages] int32, seq_lens [B] int32.
 * Outputs are written at the flattened index (o: [.., d_c], lse: [..]) when
 * sel == NULL, else compactly in selection order.
 */
void orc_decode_attn(const void* q_lat, int dql, const void* q_pe, int dqp,
                     const void* pool, int dp, const int32_t* page_table,
                     const int32_t* seq_lens, int B, int T, int H, int d_c,
                     int d_r, int page, int max_pages, double scale, int causal,
                     const int64_t* sel, int64_t n_sel, double* o, double* lse) {
    int64_t total = sel ? n_sel : (int64_t)B * T * H;
    int64_t max_len = 0;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] > max_len) max_len = seq_lens[b];
    #pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        #pragma omp for schedule(dynamic, 1)
        for (int64_t k = 0; k < total; ++k) {
            int64_t f = sel ? sel[k] : k;
            int i = (int)(f % H);
            int t = (int)((f / H) % T);
            int b = (int)(f / ((int64_t)H * T));
            int64_t n = visible_len(seq_lens[b], T, t, causal);
            decode_one(q_lat, dql, q_pe, dqp, pool, dp, page_table, n, b, t, i,
                       T, H, d_c, d_r, page, max_pages, scale, s,
                       o + k * d_c, lse + k, NULL);
        }
        free(s);
    }
}

/*
 * Training-form (unabsorbed) attention over whole sequences, every cached
 * token a query ([Mishra] "Multi-head Latent Attention": the unabsorbed form
 * is the one used in training; [llms] "Low-Rank Key-Value Joint
 * Compression" and "The Positional Problem and Decoupled RoPE" for the
 * definitions).  For sequence b, query position t and head i:
 *   k_{j,i} = [W^UK_i c_j ; k^R_j],  v_{j,i} = W^UV_i c_j
 *   s_j     = q_{t,i} . k_{j,i} * scale,   j <= t when causal, else all j < L
 *   u_{t,i} = sum_j softmax_j(s) v_{j,i},  lse_{t,i} = ln sum_j e^{s_j}
 * The same definitions as orc_naive_decode with T = L; the keys and values
 * of a sequence (they do not depend on the query) are expanded once.
 * cache [B*L, d_c+d_r] rows [c ; k^R]; q_nope [B,L,H,d_h]; q_pe [B,L,H,d_r];
 * sel lists flattened (b*L + t)*H + i rows (NULL: all), outputs compact in
 * selection order: u [rows, d_h], lse [rows].
 */
void orc_naive_prefill(const double* cache, const void* q_nope, int dqn,
                       const void* q_pe, int dqp, const void* w_uk, int dwk,
                       const void* w_uv, int dwv, int B, int L, int H, int d_h,
                       int d_c, int d_r, double scale, int causal,
                       const int64_t* sel, int64_t n_sel, double* u, double* lse) {
    int64_t width = (int64_t)d_c + d_r;
    int64_t kw = (int64_t)d_h + d_r;
    int64_t total = sel ? n_sel : (int64_t)B * L * H;
    /* expanded keys and values of every (b, j, i): [B, L, H, d_h + d_r], [B, L, H, d_h] */
    double* K = (double*)malloc(sizeof(double) * (size_t)B * L * H * kw);
    double* V = (double*)malloc(sizeof(double) * (size_t)B * L * H * d_h);
    #pragma omp parallel for collapse(3) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < L; ++j)
            for (int i = 0; i < H; ++i) {
                const double* row = cache + ((int64_t)b * L + j) * width;
                double* k = K + (((int64_t)b * L + j) * H + i) * kw;
                double* v = V + (((int64_t)b * L + j) * H + i) * d_h;
                for (int e = 0; e < d_h; ++e) {
                    double kx = 0.0, vx = 0.0;  /* (W^UK_i c_j)[e], (W^UV_i c_j)[e] */
                    int64_t wr = ((int64_t)i * d_h + e) * d_c;
                    for (int c = 0; c < d_c; ++c) {
                        kx += rd(w_uk, dwk, wr + c) * row[c];
                        vx += rd(w_uv, dwv, wr + c) * row[c];
                    }
                    k[e] = kx;
                    v[e] = vx;
                }
                for (int e = 0; e < d_r; ++e) k[d_h + e] = row[d_c + e];
            }
    #pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)L);
        #pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < total; ++r) {
            int64_t f = sel ? sel[r] : r;
            int i = (int)(f % H);
            int t = (int)((f / H) % L);
            int b = (int)(f / ((int64_t)H * L));
            int64_t n = causal ? (int64_t)t + 1 : L;
            double m = -INFINITY;
            for (int64_t j = 0; j < n; ++j) {
                const double* k = K + (((int64_t)b * L + j) * H + i) * kw;
                double acc = 0.0;
                for (int e = 0; e < d_h; ++e) acc += rd(q_nope, dqn, f * d_h + e) * k[e];
                for (int e = 0; e < d_r; ++e) acc += rd(q_pe, dqp, f * d_r + e) * k[d_h + e];
                s[j] = acc * scale;
                if (s[j] > m) m = s[j];
            }
            double l = 0.0;
            for (int64_t j = 0; j < n; ++j) l += exp(s[j] - m);
            double* ur = u + r * d_h;
            for (int e = 0; e < d_h; ++e) ur[e] = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                double a = exp(s[j] - m) / l;
                const double* v = V + (((int64_t)b * L + j) * H + i) * d_h;
                for (int e = 0; e < d_h; ++e) ur[e] += a * v[e];
            }
            lse[r] = m + log(l);
        }
        free(s);
    }
    free(K);
    free(V);
}

/*
 * Softmax attention of given per-head keys and values, every token a query:
 * the attention half of the training-form route above, on keys and values
 * already expanded ([Mishra] "Multi-head Latent Attention"; [llms] "The
 * Positional Problem and Decoupled RoPE": the RoPE key k^R_j is shared by
 * all heads).  For sequence b, position t, head i:
 *   s_j     = (q^C_{t,i} . k^C_{j,i} + q^R_{t,i} . k^R_j) * scale
 *   u_{t,i} = sum_j softmax_j(s) v_{j,i},   lse_{t,i} = ln sum_j e^{s_j}
 * over j <= t (causal) or all j < L.  q_nope, k_nope, v [B*L, H, d_h];
 * q_pe [B*L, H, d_r]; k_pe rows of k_pe_ld values, the RoPE key from
 * column k_pe_off (so that it can be read straight from cache rows).
 * sel, u, lse as in orc_naive_prefill.
 */
void orc_prefill_attn(const void* q_nope, int dqn, const void* q_pe, int dqp,
                      const void* k_nope, int dkn, const void* k_pe, int dkp,
                      int64_t k_pe_ld, int64_t k_pe_off, const void* v, int dv,
                      int B, int L, int H, int d_h, int d_r, double scale, int causal,
                      const int64_t* sel, int64_t n_sel, double* u, double* lse) {
    int64_t total = sel ? n_sel : (int64_t)B * L * H;
    #pragma omp parallel
    {
        double* sc = (double*)malloc(sizeof(double) * (size_t)L);
        #pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < total; ++r) {
            int64_t f = sel ? sel[r] : r;
            int i = (int)(f % H);
            int64_t tok = f / H;               /* b * L + t */
            int t = (int)(tok % L);
            int64_t first = tok - t;           /* the sequence's first token */
            int64_t n = causal ? t + (int64_t)1 : (int64_t)L;  /* visible keys */
            double mx = -INFINITY;
            for (int64_t j = 0; j < n; ++j) {
                int64_t kr = (first + j) * H + i;
                double acc = 0.0;
                for (int e = 0; e < d_h; ++e) acc += rd(q_nope, dqn, f * d_h + e) * rd(k_nope, dkn, kr * d_h + e);
                for (int e = 0; e < d_r; ++e)
                    acc += rd(q_pe, dqp, f * d_r + e) * rd(k_pe, dkp, (first + j) * k_pe_ld + k_pe_off + e);
                sc[j] = acc * scale;
                if (sc[j] > mx) mx = sc[j];
            }
            double den = 0.0;
            for (int64_t j = 0; j < n; ++j) den += exp(sc[j] - mx);
            double* ur = u + r * d_h;
            for (int e = 0; e < d_h; ++e) ur[e] = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                double w = exp(sc[j] - mx) / den;
                int64_t vr = (first + j) * H + i;
                for (int e = 0; e < d_h; ++e) ur[e] += w * rd(v, dv, vr * d_h + e);
            }
            lse[r] = mx + log(den);
        }
        free(sc);
    }
}

/*
 * Sensitivity of o to rounding the attention weights (test infrastructure,
 * not a step of the method).  For every listed (b, t, i) and latent column c
 *     D[c] = sum_j a_j |c_j[c] - o[c]|
 * with a_j and o of decode_one.  If every weight is perturbed to
 * a_j (1 + e_j) and the weights renormalised, o moves by
 *     sum_j a_j (e_j - ebar) c_j / (1 + ebar) = sum_j a_j e_j (c_j - o) / (1 + ebar)
 * (ebar = sum_j a_j e_j), so |e_j| <= u moves o[c] by at most
 * u / (1 - u) * D[c].  Rounding the weights to bf16 has u = 2^-8.
 * sel as in orc_decode_attn (NULL: every row); D [rows, d_c].
 */
void orc_weight_spread(const void* q_lat, int dql, const void* q_pe, int dqp,
                       const void* pool, int dp, const int32_t* page_table,
                       const int32_t* seq_lens, int B, int T, int H, int d_c,
                       int d_r, int page, int max_pages, double scale, int causal,
                       const int64_t* sel, int64_t n_sel, double* D) {
    int64_t total = sel ? n_sel : (int64_t)B * T * H;
    int64_t max_len = 0;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] > max_len) max_len = seq_lens[b];
    int64_t width = (int64_t)d_c + d_r;
    #pragma omp parallel
    {
        size_t cap = (size_t)(max_len > 0 ? max_len : 1);
        double* s = (double*)malloc(sizeof(double) * cap);
        double* a = (double*)malloc(sizeof(double) * cap);
        double* o = (double*)malloc(sizeof(double) * (size_t)d_c);
        #pragma omp for schedule(dynamic, 1)
        for (int64_t k = 0; k < total; ++k) {
            int64_t f = sel ? sel[k] : k;
            int i = (int)(f % H);
            int t = (int)((f / H) % T);
            int b = (int)(f / ((int64_t)H * T));
            int64_t n = visible_len(seq_lens[b], T, t, causal);
            double lse;
            decode_one(q_lat, dql, q_pe, dqp, pool, dp, page_table, n, b, t, i,
                       T, H, d_c, d_r, page, max_pages, scale, s, o, &lse, a);
            double* dst = D + k * d_c;
            for (int c = 0; c < d_c; ++c) dst[c] = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                int64_t pg = page_table[(int64_t)b * max_pages + j / page];
                int64_t row = (pg * page + j % page) * width;
                for (int c = 0; c < d_c; ++c)
                    dst[c] += a[j] * fabs(rd(pool, dp, row + c) - o[c]);
            }
        }
        free(s);
        free(a);
        free(o);
    }
}

/*
 * Attention weights a_j of one (b, t, i): the softmax row the decode uses.
 * [Zhang] "Value absorption": softmax over the scaled scores gives A(i, j).
 * a_out receives the n visible weights; returns n.
 */
int64_t orc_attention_weights(const void* q_lat, int dql, const void* q_pe, int dqp,
                              const void* pool, int dp, const int32_t* page_table,
                              const int32_t* seq_lens, int T, int H, int d_c,
                              int d_r, int page, int max_pages, double scale,
                              int causal, int b, int t, int i, double* a_out) {
    int64_t n = visible_len(seq_lens[b], T, t, causal);
    double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double* o_row = (double*)malloc(sizeof(double) * (size_t)d_c);
    double lse;
    decode_one(q_lat, dql, q_pe, dqp, pool, dp, page_table, n, b, t, i, T, H,
               d_c, d_r, page, max_pages, scale, s, o_row, &lse, a_out);
    free(s);
    free(o_row);
    return n;
}

/*
 * Merge of partial results over disjoint pieces of one softmax:
 *   lse = ln sum_s exp(lse_s),  o = sum_s exp(lse_s - lse) o_s.
 * A piece with lse_s = -inf has weight 0; if every piece is empty the
 * result is o = 0, lse = -inf.
 * o_part [S, N, d_c] (dtype dpo), lse_part [S, N] (dtype dpl) -> o [N, d_c], lse [N].
 */
void orc_combine(const void* o_part, int dpo, const void* lse_part, int dpl,
                 int S, int64_t N, int d_c, double* o, double* lse) {
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) {
        double m = -INFINITY;
        for (int s = 0; s < S; ++s) {
            double v = rd(lse_part, dpl, (int64_t)s * N + r);
            if (v > m) m = v;
        }
        for (int c = 0; c < d_c; ++c) o[r * d_c + c] = 0.0;
        if (m == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int s = 0; s < S; ++s) sum += exp(rd(lse_part, dpl, (int64_t)s * N + r) - m);
        double L = m + log(sum);
        for (int s = 0; s < S; ++s) {
            double w = exp(rd(lse_part, dpl, (int64_t)s * N + r) - L);
            if (w == 0.0) continue;
            for (int c = 0; c < d_c; ++c)
                o[r * d_c + c] += w * rd(o_part, dpo, ((int64_t)s * N + r) * d_c + c);
        }
        lse[r] = L;
    }
}

/*
 * Output side: u_i = W^UV_i o_i (d_c -> d_h), out = W^O concat_i u_i.
 * [llms] "Value Output Absorption"; [Zhang] "Value absorption": W^UV is
 * applied once to the latent-weighted sum, and kept apart from W^O.
 * o [R,H,d_c], w_uv [H,d_h,d_c], w_o [d, H*d_h] -> out [R,d]; u (optional) [R,H*d_h].
 */
void orc_out_proj(const void* o, int dov, const void* w_uv, int dwu,
                  const void* w_o, int dwo, int R, int H, int d_h, int d_c,
                  int d, double* out, double* u_out) {
    int64_t hd = (int64_t)H * d_h;
    double* u = (double*)malloc(sizeof(double) * (size_t)R * (size_t)hd);
    #pragma omp parallel for collapse(2) schedule(static)
    for (int r = 0; r < R; ++r)
        for (int i = 0; i < H; ++i)
            for (int e = 0; e < d_h; ++e) {
                double acc = 0.0;
                int64_t wrow = ((int64_t)i * d_h + e) * d_c;
                int64_t orow = ((int64_t)r * H + i) * d_c;
                for (int c = 0; c < d_c; ++c)
                    acc += rd(w_uv, dwu, wrow + c) * rd(o, dov, orow + c);
                u[(int64_t)r * hd + (int64_t)i * d_h + e] = acc;
            }
    #pragma omp parallel for collapse(2) schedule(static)
    for (int r = 0; r < R; ++r)
        for (int n = 0; n < d; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < hd; ++k) acc += rd(w_o, dwo, (int64_t)n * hd + k) * u[(int64_t)r * hd + k];
            out[(int64_t)r * d + n] = acc;
        }
    if (u_out) memcpy(u_out, u, sizeof(double) * (size_t)R * (size_t)hd);
    free(u);
}

/* ------------------------------------- producer step (model -> cache) */

/*
 * From hidden states to the quantities the decode path consumes, for
 * sequences of L tokens at positions 0..L-1 (contiguous cache):
 *   c_j   = W^DKV h_j                       [Mishra] "Step 1: a low-rank latent"
 *   k^R_j = RoPE(W^KR h_j, j)               [Zhang] "Decoupled RoPE"; [llms]
 *                                            "The Positional Problem and Decoupled RoPE"
 *   q     = W^Q h_q, head i = [q^C_i ; q^R_i], q^R_i rotated at the query
 *           position qpos                   [llms] ("q_{t,i} = [q^C ; q^R]")
 * The query token is h[b, qpos].  W^Q is [H*(d_h+d_r) x d] with head i owning
 * rows i*(d_h+d_r) .. +d_h+d_r-1, content rows first (a reading: the pages
 * concatenate q = [q^C ; q^R] but print no single W^Q).
 * h [B,L,d]; w_dkv [d_c,d]; w_kr [d_r,d]; w_q [H*(d_h+d_r), d]
 * -> cache [B*L, d_c+d_r] (row b*L+j), q_nope [B,H,d_h], q_pe [B,H,d_r].
 */
void orc_project(const void* h, int dh_t, const void* w_dkv, int dw1,
                 const void* w_kr, int dw2, const void* w_q, int dw3, int B,
                 int L, int d, int H, int d_h, int d_c, int d_r, int qpos,
                 double rope_base, double* cache, double* q_nope, double* q_pe) {
    int64_t width = (int64_t)d_c + d_r;
    #pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < L; ++j) {
            int64_t hrow = ((int64_t)b * L + j) * d;
            double* row = cache + ((int64_t)b * L + j) * width;
            for (int c = 0; c < d_c; ++c) {
                double acc = 0.0;
                for (int k = 0; k < d; ++k) acc += rd(w_dkv, dw1, (int64_t)c * d + k) * rd(h, dh_t, hrow + k);
                row[c] = acc;
            }
            for (int e = 0; e < d_r; ++e) {
                double acc = 0.0;
                for (int k = 0; k < d; ++k) acc += rd(w_kr, dw2, (int64_t)e * d + k) * rd(h, dh_t, hrow + k);
                row[d_c + e] = acc;
            }
            orc_rope(row + d_c, d_r, (double)j, rope_base);
        }
    int64_t qw = (int64_t)d_h + d_r;
    for (int b = 0; b < B; ++b) {
        int64_t hrow = ((int64_t)b * L + qpos) * d;
        for (int i = 0; i < H; ++i) {
            for (int e = 0; e < qw; ++e) {
                double acc = 0.0;
                int64_t wrow = ((int64_t)i * qw + e) * d;
                for (int k = 0; k < d; ++k) acc += rd(w_q, dw3, wrow + k) * rd(h, dh_t, hrow + k);
                if (e < d_h) q_nope[((int64_t)b * H + i) * d_h + e] = acc;
                else q_pe[((int64_t)b * H + i) * d_r + (e - d_h)] = acc;
            }
            orc_rope(q_pe + ((int64_t)b * H + i) * d_r, d_r, (double)qpos, rope_base);
        }
    }
}

/* ---------------------------------------------------- naive route */

/*
 * Naive MLA decode: the cached latents are expanded to per-head keys and
 * values every step and ordinary softmax attention runs on them.
 *   k_{j,i} = [W^UK_i c_j ; k^R_j],  v_{j,i} = W^UV_i c_j
 *       ([llms] "Low-Rank Key-Value Joint Compression" and "The Positional
 *       Problem and Decoupled RoPE": q_{t,i} = [q^C ; q^R], k_{j,i} = [k^C ; k^R])
 *   s_ij = q_i . k_{j,i} * scale;  a = softmax_j(s)
 *   u_i  = sum_j a_ij v_{j,i};     out = W^O concat_i u_i
 * Absorption ([Mishra] "Step 2", [Zhang] "Matrix absorption", [llms]
 * "Inference Optimization: Weight Matrix Absorption") is an exact
 * reassociation of this; the oracle keeps both routes so that one can be
 * checked against the other.
 * cache [B*L, d_c+d_r] contiguous per sequence, q_nope [B,T,H,d_h],
 * q_pe [B,T,H,d_r]; query t sees positions 0..n_t-1 (visible_len with len L).
 * Outputs: u [B,T,H,d_h], out [B,T,d] (out may be NULL when w_o is NULL).
 */
void orc_naive_decode(const double* cache, const void* q_nope, int dqn,
                      const void* q_pe, int dqp, const void* w_uk, int dwk,
                      const void* w_uv, int dwv, const void* w_o, int dwo,
                      int B, int T, int L, int H, int d_h, int d_c, int d_r,
                      int d, double scale, int causal, double* u, double* out) {
    int64_t width = (int64_t)d_c + d_r;
    #pragma omp parallel
    {
        double* k = (double*)malloc(sizeof(double) * (size_t)L * (size_t)(d_h + d_r));
        double* v = (double*)malloc(sizeof(double) * (size_t)L * (size_t)d_h);
        double* s = (double*)malloc(sizeof(double) * (size_t)L);
        #pragma omp for collapse(3) schedule(dynamic, 1)
        for (int b = 0; b < B; ++b)
            for (int t = 0; t < T; ++t)
                for (int i = 0; i < H; ++i) {
                    int64_t n = visible_len(L, T, t, causal);
                    for (int64_t j = 0; j < n; ++j) {
                        const double* row = cache + ((int64_t)b * L + j) * width;
                        for (int e = 0; e < d_h; ++e) {
                            double ak = 0.0, av = 0.0;
                            int64_t wrow = ((int64_t)i * d_h + e) * d_c;
                            for (int c = 0; c < d_c; ++c) {
                                ak += rd(w_uk, dwk, wrow + c) * row[c];
                                av += rd(w_uv, dwv, wrow + c) * row[c];
                            }
                            k[j * (d_h + d_r) + e] = ak;
                            v[j * d_h + e] = av;
                        }
                        for (int e = 0; e < d_r; ++e) k[j * (d_h + d_r) + d_h + e] = row[d_c + e];
                    }
                    int64_t qrow = ((int64_t)b * T + t) * H + i;
                    double m = -INFINITY;
                    for (int64_t j = 0; j < n; ++j) {
                        double acc = 0.0;
                        for (int e = 0; e < d_h; ++e) acc += rd(q_nope, dqn, qrow * d_h + e) * k[j * (d_h + d_r) + e];
                        for (int e = 0; e < d_r; ++e) acc += rd(q_pe, dqp, qrow * d_r + e) * k[j * (d_h + d_r) + d_h + e];
                        s[j] = acc * scale;
                        if (s[j] > m) m = s[j];
                    }
                    double l = 0.0;
                    for (int64_t j = 0; j < n; ++j) l += exp(s[j] - m);
                    double* ui = u + qrow * d_h;
                    for (int e = 0; e < d_h; ++e) ui[e] = 0.0;
                    for (int64_t j = 0; j < n; ++j) {
                        double a = exp(s[j] - m) / l;
                        for (int e = 0; e < d_h; ++e) ui[e] += a * v[j * d_h + e];
                    }
                }
        free(k);
        free(v);
        free(s);
    }
    if (!out || !w_o) return;
    int64_t hd = (int64_t)H * d_h;
    #pragma omp parallel for collapse(2) schedule(static)
    for (int r = 0; r < B * T; ++r)
        for (int n = 0; n < d; ++n) {
            double acc = 0.0;
            for (int64_t kk = 0; kk < hd; ++kk) acc += rd(w_o, dwo, (int64_t)n * hd + kk) * u[(int64_t)r * hd + kk];
            out[(int64_t)r * d + n] = acc;
        }
}
