"""Pins of the fp64 oracle to facts outside itself.

Each ``pin_*`` function takes an oracle library handle (``oracle.load()`` or
a deliberately broken build of it) and raises AssertionError when the oracle
disagrees with what the pages print, a closed form, an invariant, or a
library routine (torch CPU fp64 ``scaled_dot_product_attention``, matmul,
``logsumexp``).  ``test_oracle_pins.py`` runs them against the real oracle;
``test_oracle_mutants.py`` checks that planted mistakes in the oracle make at
least one of them fail.

Pages cited:
  [Mishra]  "Multi-head Latent Attention", Neel Mishra
  [Zhang]   zhangchitc.github.io, Multi-Head Latent Attention post
  [llms]    "Multi-Head Latent Attention: How Low-Rank KV Compression Scales
            LLM Serving"
  [DataMListic] "Multi-Head Latent Attention (MLA) - Explained"
"""

from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle
from mla_latent_kv_71_b300 import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "page_numbers.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _small_case(B=3, T=1, H=4, d_c=32, d_r=8, lens=(1, 63, 130), seed=5, page=16,
                dtype=torch.float64, causal=None):
    return workloads.decode_case(B, T, H, d_c, d_r, list(lens), page=page, seed=seed,
                                 dtype=dtype, d_h=16, causal=causal)


def _gather_kv(case, b):
    """Logical cache rows of sequence b, gathered through the page table."""
    page = case.pool.shape[1]
    n = int(case.seq_lens[b])
    j = torch.arange(n)
    pages = case.page_table[b, j // page].long()
    return case.pool[pages, j % page].to(torch.float64)  # [n, d_c + d_r]


# ----------------------------------------------------------------- accounting

def pin_cache_accounting(lib):
    """(b) cache sizes per token per layer against the printed numbers."""
    g = _golden()
    a = g["accounting_table"]
    nums = oracle.cache_numbers(a["h"], a["d_h"], a["h_kv"], a["d_c"], a["d_r"], lib=lib)
    assert nums["MHA"] == a["MHA"] and nums["GQA"] == a["GQA"], nums
    assert nums["MQA"] == a["MQA"] and nums["MLA"] == a["MLA"], nums
    m = g["mha_vs_latent"]
    assert nums["MLA_latent"] == m["MLA_latent"]
    assert nums["MHA"] // nums["MLA_latent"] == m["ratio"] and nums["MHA"] % nums["MLA_latent"] == 0
    r = g["mla_with_rope_key"]
    assert round(nums["MHA"] / nums["MLA"]) == r["ratio_approx"]
    p = g["reductions_percent"]
    assert round(100 * (1 - nums["MLA"] / nums["MHA"]), 1) == p["vs_MHA"]
    assert round(100 * (1 - nums["MLA"] / nums["GQA"]), 1) == p["vs_GQA8"]
    e = g["eight_heads_of_64"]
    assert oracle.cache_numbers(e["h"], e["d_h"], 1, 1, 0, lib=lib)["MHA"] > e["more_than"]


def pin_absorption_cost(lib):
    """The n = 100 count of the two multiplication orders, as printed."""
    c = _golden()["absorption_cost"]
    key, query = oracle.score_cost(c["n"], c["hd"], c["d_c"], lib=lib)
    assert key == eval(c["key_side"], {}) and query == eval(c["query_side"], {})
    assert round(key / query) == c["ratio_approx"]


# ----------------------------------------------------------------------- RoPE

def pin_rope(lib):
    """RoPE closed forms: identity at 0, the per-pair angle, norm, relativity."""
    rng = np.random.default_rng(0)
    x = rng.standard_normal(16)
    assert np.array_equal(oracle.rope(x, 0, lib=lib), x)
    # pair k rotates by pos * base^(-2k/d_r): d_r = 4, base 10000 -> pair 1 at 1/100
    y = oracle.rope([0.0, 0.0, 1.0, 0.0], 100, lib=lib)
    assert np.allclose(y, [0.0, 0.0, math.cos(1.0), math.sin(1.0)], atol=1e-15, rtol=0)
    y = oracle.rope([0.0, 1.0], 0.5, lib=lib)  # pair 0: angle = pos
    assert np.allclose(y, [-math.sin(0.5), math.cos(0.5)], atol=1e-15, rtol=0)
    assert abs(np.linalg.norm(oracle.rope(x, 37, lib=lib)) - np.linalg.norm(x)) < 1e-12
    q, k = rng.standard_normal(16), rng.standard_normal(16)
    d1 = oracle.rope(q, 50, lib=lib) @ oracle.rope(k, 20, lib=lib)
    d2 = oracle.rope(q, 1050, lib=lib) @ oracle.rope(k, 1020, lib=lib)
    assert abs(d1 - d2) < 1e-9 * max(1.0, abs(d1))
    # at the long-context positions the cache write uses (up to 131071):
    # rotations compose, R(a) R(b) = R(a + b), and the relative score holds
    x64 = rng.standard_normal(64)
    a, b = 100000, 31071
    assert np.abs(oracle.rope(oracle.rope(x64, a, lib=lib), b, lib=lib)
                  - oracle.rope(x64, a + b, lib=lib)).max() < 1e-9
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    d1 = oracle.rope(q, 7, lib=lib) @ oracle.rope(k, 3, lib=lib)
    d2 = oracle.rope(q, 131071, lib=lib) @ oracle.rope(k, 131067, lib=lib)
    assert abs(d1 - d2) < 1e-8 * max(1.0, abs(d1))


# ------------------------------------------------------------ tiny fp32 model

def _tiny_routes(lib):
    m = workloads.tiny_model(seed=0)
    B, L, H, d_h, d_c = m["B"], m["L"], m["H"], m["d_h"], m["d_c"]
    h = m["h"].to(torch.float64)
    cache, q_nope, q_pe = oracle.project(h, m["w_dkv"], m["w_kr"], m["w_q"], H, d_h,
                                         qpos=L - 1, lib=lib)
    u_n, out_n = oracle.naive_decode(cache, q_nope[:, None], q_pe[:, None], m["w_uk"],
                                     m["w_uv"], m["w_o"], L, m["scale"], lib=lib)
    q_lat = oracle.absorb_q(q_nope, m["w_uk"], lib=lib)                    # [B,H,d_c]
    pool = cache.reshape(B * L // 64, 64, cache.shape[1])
    table = np.arange(B * L // 64, dtype=np.int32).reshape(B, L // 64)
    o, lse = oracle.decode_attn(q_lat[:, None], q_pe[:, None], pool, table,
                                np.full(B, L, np.int32), m["scale"], lib=lib)
    out_a, u_a = oracle.out_proj(o[:, 0], m["w_uv"], m["w_o"], lib=lib)
    return m, cache, q_nope, q_pe, u_n, out_n, u_a, out_a, o, lse


def pin_naive_equals_absorbed(lib):
    """(a) the associativity identity on the tiny model: both routes agree.

    [Mishra] 'Step 2: absorb the up-projections'; [Zhang] 'Matrix absorption'
    and 'Value absorption'; [llms] 'Query Key Absorption', 'Value Output
    Absorption': reassociating the products changes no result.
    """
    m, cache, q_nope, q_pe, u_n, out_n, u_a, out_a, o, lse = _tiny_routes(lib)
    B, H, d_h = m["B"], m["H"], m["d_h"]
    assert _rel(u_a.reshape(B, H, d_h), u_n[:, 0]) < 1e-12
    assert _rel(out_a, out_n[:, 0]) < 1e-12
    assert np.abs(out_n).max() > 1e-3  # not a vacuous zero



def pin_naive_equals_absorbed_at_model_widths(lib):
    """(a) again, at the DeepSeek-V2/V3 widths the GPU path runs (d_c = 512,
    d_h = 128, d_r = 64, d = 7168), with two causal query tokens, bf16 inputs
    and a paged, permuted cache on the absorbed side.

    A subsample (2 sequences of 130 rows, 4 heads) keeps the naive route,
    which expands K and V for every head, to a second of CPU.  Same passages
    as the tiny-model check: reassociating the products changes no result.
    """
    B, T, H, d_h, d_c, d_r, d, L = 2, 2, 4, 128, 512, 64, 7168, 130
    case = workloads.decode_case(B, T, H, d_c, d_r, [L] * B, seed=21, d_h=d_h)
    w_uk, w_uv, w_o = workloads.projection_weights(H, d_h, d_c, d, seed=22)
    q_nope = workloads.q_nope(B, T, H, d_h, seed=23)
    cache = torch.cat([_gather_kv(case, b) for b in range(B)]).numpy()  # [B*L, d_c+d_r]
    u_n, out_n = oracle.naive_decode(cache, q_nope, case.q_pe, w_uk, w_uv, w_o, L,
                                     case.scale, causal=True, lib=lib)
    q_lat = oracle.absorb_q(q_nope.reshape(B * T, H, d_h), w_uk, lib=lib)
    o, lse = oracle.decode_attn(q_lat.reshape(B, T, H, d_c), case.q_pe, case.pool,
                                case.page_table, case.seq_lens, case.scale, causal=True,
                                lib=lib)
    out_a, u_a = oracle.out_proj(o.reshape(B * T, H, d_c), w_uv, w_o, lib=lib)
    assert _rel(u_a.reshape(u_n.shape), u_n) < 1e-12
    assert _rel(out_a.reshape(out_n.shape), out_n) < 1e-12
    assert np.abs(out_n).max() > 1e-2  # not a vacuous zero


def pin_naive_vs_library_sdpa(lib):
    """The naive route's attention equals torch's fp64 SDPA on the expanded K, V.

    Keys and values are expanded per the pages' definitions
    (k = [W^UK c ; k^R], v = W^UV c: [llms] 'Low-Rank Key-Value Joint
    Compression', 'The Positional Problem and Decoupled RoPE') and handed to
    the library routine with scale 1/sqrt(d_h + d_r) ([Zhang] 'Value absorption').
    """
    m, cache, q_nope, q_pe, u_n, *_ = _tiny_routes(lib)
    B, L, H, d_h, d_c = m["B"], m["L"], m["H"], m["d_h"], m["d_c"]
    c = torch.from_numpy(cache[:, :d_c]).reshape(B, L, d_c)
    kr = torch.from_numpy(cache[:, d_c:]).reshape(B, L, -1)
    w_uk = m["w_uk"].double()
    w_uv = m["w_uv"].double()
    k_c = torch.einsum("hec,blc->bhle", w_uk, c)
    v = torch.einsum("hec,blc->bhle", w_uv, c)
    k = torch.cat([k_c, kr[:, None].expand(B, H, L, kr.shape[-1])], dim=-1)
    q = torch.cat([torch.from_numpy(q_nope), torch.from_numpy(q_pe)], dim=-1)[:, :, None]
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=m["scale"])
    assert _rel(u_n[:, 0], ref[:, :, 0].numpy()) < 1e-12


def pin_project_vs_library(lib):
    """Projections equal library matmuls; the query's RoPE lane is rotated at L-1."""
    m = workloads.tiny_model(seed=0)
    B, L, H, d_h, d_c, d_r = m["B"], m["L"], m["H"], m["d_h"], m["d_c"], m["d_r"]
    h = m["h"].double()
    cache, q_nope, q_pe = oracle.project(h, m["w_dkv"], m["w_kr"], m["w_q"], H, d_h,
                                         qpos=L - 1, lib=lib)
    c_ref = (h @ m["w_dkv"].double().T).reshape(B * L, d_c)
    assert _rel(cache[:, :d_c], c_ref.numpy()) < 1e-13
    kr_raw = (h @ m["w_kr"].double().T).reshape(B * L, d_r).numpy()
    assert abs(np.linalg.norm(cache[:, d_c:]) - np.linalg.norm(kr_raw)) < 1e-9
    assert np.allclose(cache[0, d_c:], kr_raw[0], atol=1e-13)  # position 0: no rotation
    j = 5
    assert np.allclose(cache[j, d_c:], oracle.rope(kr_raw[j], j, lib=lib), atol=1e-13)
    qf = (h[:, L - 1] @ m["w_q"].double().T).reshape(B, H, d_h + d_r).numpy()
    assert _rel(q_nope, qf[..., :d_h]) < 1e-13
    assert np.allclose(q_pe[1, 3], oracle.rope(qf[1, 3, d_h:], L - 1, lib=lib), atol=1e-13)


def pin_position_shift_invariance(lib):
    """Shifting every position by the same amount leaves the output unchanged.

    RoPE encodes relative position ([Mishra] 'Step 3: RoPE breaks it':
    the rotation depends on j - t only).
    """
    m = workloads.tiny_model(seed=0)
    B, L, H, d_h, d_c, d_r = m["B"], m["L"], m["H"], m["d_h"], m["d_c"], m["d_r"]
    h = m["h"].double()
    outs = []
    for pad in (0, 17):
        hp = torch.cat([torch.zeros(B, pad, h.shape[2], dtype=h.dtype), h], dim=1)
        cache, q_nope, q_pe = oracle.project(hp, m["w_dkv"], m["w_kr"], m["w_q"], H, d_h,
                                             qpos=pad + L - 1, lib=lib)
        cache = cache.reshape(B, pad + L, -1)[:, pad:].reshape(B * L, -1)
        u, out = oracle.naive_decode(cache, q_nope[:, None], q_pe[:, None], m["w_uk"],
                                     m["w_uv"], m["w_o"], L, m["scale"], lib=lib)
        outs.append(out)
    assert _rel(outs[1], outs[0]) < 1e-11


# ---------------------------------------------------------------- paged decode

def pin_decode_vs_library_sdpa(lib):
    """Paged absorbed decode equals torch fp64 SDPA on the gathered rows.

    Scores use q = [q_lat ; q_pe] against [c ; k^R] and the values are the
    latents c ([llms] 'Query Key Absorption', 'Value Output Absorption');
    causal queries see positions 0..len-T+t.  lse equals torch.logsumexp of
    the scaled scores.
    """
    for T in (1, 2):
        case = _small_case(T=T, lens=(1, 63, 130) if T == 1 else (2, 64, 131), seed=7 + T)
        o, lse = oracle.decode_attn(case.q_lat, case.q_pe, case.pool, case.page_table,
                                    case.seq_lens, case.scale, causal=case.causal, lib=lib)
        d_c = case.q_lat.shape[3]
        for b in range(case.q_lat.shape[0]):
            rows = _gather_kv(case, b)
            n = rows.shape[0]
            q = torch.cat([case.q_lat[b], case.q_pe[b]], dim=-1).double().transpose(0, 1)
            k = rows[None].expand(q.shape[0], n, rows.shape[1])
            v = rows[None, :, :d_c].expand(q.shape[0], n, d_c)
            mask = torch.ones(T, n, dtype=torch.bool)
            for t in range(T):
                mask[t, n - (T - 1 - t):] = False
            ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask,
                                                                   scale=case.scale)
            assert _rel(o[b].transpose(1, 0, 2), ref.numpy()) < 1e-12
            s = (q @ k.transpose(1, 2)) * case.scale
            s = s.masked_fill(~mask, float("-inf"))
            ref_lse = torch.logsumexp(s, dim=-1)  # [H, T]
            assert np.abs(lse[b].T - ref_lse.numpy()).max() < 1e-12


def pin_decode_closed_forms(lib):
    """L = 1 gives o = c_0, lse = s_0; q = 0 gives the mean and ln L; equal rows."""
    case = _small_case(lens=(1, 50, 64), seed=11)
    d_c = case.q_lat.shape[3]
    o, lse = oracle.decode_attn(case.q_lat, case.q_pe, case.pool, case.page_table,
                                case.seq_lens, case.scale, lib=lib)
    row0 = _gather_kv(case, 0)[0]
    assert np.array_equal(o[0, 0], np.broadcast_to(row0[:d_c].numpy(), o[0, 0].shape))
    s0 = (torch.cat([case.q_lat[0, 0], case.q_pe[0, 0]], -1).double() @ row0) * case.scale
    assert np.abs(lse[0, 0] - s0.numpy()).max() < 1e-12
    zero = _small_case(lens=(1, 50, 64), seed=11)
    zero.q_lat.zero_()
    zero.q_pe.zero_()
    o, lse = oracle.decode_attn(zero.q_lat, zero.q_pe, zero.pool, zero.page_table,
                                zero.seq_lens, zero.scale, lib=lib)
    for b, n in enumerate((1, 50, 64)):
        mean = _gather_kv(zero, b)[:, :d_c].mean(0).numpy()
        assert np.abs(o[b, 0] - mean).max() < 1e-13
        assert np.abs(lse[b, 0] - math.log(n)).max() < 1e-13
    same = _small_case(lens=(5, 40, 64), seed=12)
    same.pool[:] = same.pool[0, 0]
    o, lse = oracle.decode_attn(same.q_lat, same.q_pe, same.pool, same.page_table,
                                same.seq_lens, same.scale, lib=lib)
    assert np.abs(o - same.pool[0, 0, :d_c].numpy()).max() < 1e-13


def pin_softmax_rows_sum_to_one(lib):
    """(c) the softmax row of every (b, t, i) sums to one ([Zhang] 'Value absorption')."""
    case = _small_case(T=2, lens=(3, 64, 129), seed=13)
    B, T, H = case.q_lat.shape[:3]
    for b in range(B):
        for t in range(T):
            for i in range(H):
                a = oracle.attention_weights(case.q_lat, case.q_pe, case.pool, case.page_table,
                                             case.seq_lens, case.scale, b, t, i, causal=True,
                                             lib=lib)
                assert len(a) == int(case.seq_lens[b]) - (T - 1 - t)
                assert abs(a.sum() - 1.0) < 1e-14 and (a >= 0).all()



def pin_fp64_rounding_is_negligible(lib):
    """The oracle's fp64 rounding is far below every tolerance it serves.

    One 4096-row sequence with 1 % of its latent rows scaled by 8 (the
    long-context workload's hot rows) is decoded by the oracle and, from the
    definition (softmax of the scaled scores, latent-weighted sum, natural-log
    lse), in numpy's extended precision (64-bit significand on x86): the two
    agree to about 1e-14, eleven orders of magnitude inside the bf16 bars.
    """
    case = workloads.decode_case(1, 1, 2, 512, 64, [4096], seed=24, hot_frac=0.01)
    o, lse = oracle.decode_attn(case.q_lat, case.q_pe, case.pool, case.page_table,
                                case.seq_lens, case.scale, lib=lib)
    ld = np.longdouble
    rows = _gather_kv(case, 0).numpy().astype(ld)                           # [n, 576]
    q = torch.cat([case.q_lat[0, 0], case.q_pe[0, 0]], -1).double().numpy().astype(ld)
    s = (q @ rows.T) * ld(case.scale)                                       # [H, n]
    m = s.max(axis=1, keepdims=True)
    w = np.exp(s - m)
    ref_o = (w @ rows[:, :512]) / w.sum(axis=1, keepdims=True)
    ref_lse = m[:, 0] + np.log(w.sum(axis=1))
    assert np.finfo(ld).nmant >= 63  # an extended type, not a second double
    assert float(np.abs(o[0, 0] - ref_o).max() / np.abs(ref_o).max()) < 1e-13
    assert float(np.abs(lse[0, 0] - ref_lse).max()) < 1e-12


def pin_page_permutation_invariance(lib):
    """Where the pages sit in the pool does not change the result (exactly)."""
    case = _small_case(lens=(17, 100, 64), seed=14)
    o1, l1 = oracle.decode_attn(case.q_lat, case.q_pe, case.pool, case.page_table,
                                case.seq_lens, case.scale, lib=lib)
    P = case.pool.shape[0]
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P)
    pool2 = case.pool[perm]
    table2 = case.page_table.clone()
    valid = table2 >= 0
    table2[valid] = inv[table2[valid].long()].to(torch.int32)
    o2, l2 = oracle.decode_attn(case.q_lat, case.q_pe, pool2, table2, case.seq_lens,
                                case.scale, lib=lib)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def pin_combine_split_identity(lib):
    """Decoding disjoint page ranges and merging them reproduces the full decode.

    Also covers an empty piece (lse = -inf, weight 0) and an all-empty row.
    """
    case = _small_case(lens=(130, 64, 200), seed=15)
    B, T, H, d_c = case.q_lat.shape
    o_full, l_full = oracle.decode_attn(case.q_lat, case.q_pe, case.pool, case.page_table,
                                        case.seq_lens, case.scale, lib=lib)
    page = case.pool.shape[1]
    cuts = [0, 2, 5, case.page_table.shape[1]]  # page boundaries of 3 pieces
    parts_o, parts_l = [], []
    for s in range(3):
        lens = []
        table = torch.full_like(case.page_table, -1)
        for b in range(B):
            n_pg = math.ceil(int(case.seq_lens[b]) / page)
            p0, p1 = min(cuts[s], n_pg), min(cuts[s + 1], n_pg)
            lens.append(max(0, min(int(case.seq_lens[b]), p1 * page) - p0 * page))
            table[b, :p1 - p0] = case.page_table[b, p0:p1]
        o, l = oracle.decode_attn(case.q_lat, case.q_pe, case.pool, table,
                                  np.array(lens, np.int32), case.scale, lib=lib)
        parts_o.append(o.reshape(-1, d_c))
        parts_l.append(l.reshape(-1))
    assert np.isneginf(parts_l[2][H:2 * H]).all()  # sequence 1 has no third piece
    o, l = oracle.combine(np.stack(parts_o), np.stack(parts_l), lib=lib)
    assert _rel(o, o_full.reshape(-1, d_c)) < 1e-13
    assert np.abs(l - l_full.reshape(-1)).max() < 1e-12
    o0, l0 = oracle.combine(np.zeros((2, 1, 4)), np.full((2, 1), -np.inf), lib=lib)
    assert np.isneginf(l0).all() and (o0 == 0).all()


def pin_empty_sequence(lib):
    """A sequence that sees no cached position yields o = 0 and lse = -inf."""
    case = _small_case(lens=(0, 5, 64), seed=16)
    o, lse = oracle.decode_attn(case.q_lat, case.q_pe, case.pool, case.page_table,
                                case.seq_lens, case.scale, lib=lib)
    assert (o[0] == 0).all() and np.isneginf(lse[0]).all()
    assert np.isfinite(lse[1:]).all()


def pin_out_proj_vs_library(lib):
    """out = W^O concat_i(W^UV_i o_i) equals library matmuls."""
    g = torch.Generator().manual_seed(21)
    R, H, d_h, d_c, d = 3, 4, 8, 16, 24
    o = torch.randn(R, H, d_c, generator=g, dtype=torch.float64)
    w_uv = torch.randn(H, d_h, d_c, generator=g, dtype=torch.float64)
    w_o = torch.randn(d, H * d_h, generator=g, dtype=torch.float64)
    out, u = oracle.out_proj(o, w_uv, w_o, lib=lib)
    u_ref = torch.bmm(w_uv, o.transpose(0, 1).transpose(1, 2))  # [H, d_h, R]
    u_ref = u_ref.permute(2, 0, 1).reshape(R, H * d_h)
    assert _rel(u, u_ref.numpy()) < 1e-14
    assert _rel(out, (u_ref @ w_o.T).numpy()) < 1e-14
    qn = torch.randn(R, H, d_h, generator=g, dtype=torch.float64)
    w_uk = torch.randn(H, d_h, d_c, generator=g, dtype=torch.float64)
    q_lat = oracle.absorb_q(qn, w_uk, lib=lib)
    ref = torch.bmm(qn.transpose(0, 1), w_uk).transpose(0, 1)  # [R, H, d_c]
    assert _rel(q_lat, ref.numpy()) < 1e-14


def pin_bf16_widening(lib):
    """bf16 inputs are widened exactly: same result as the fp64 copy of them."""
    case = _small_case(lens=(9, 70, 64), seed=17, dtype=torch.bfloat16)
    o1, l1 = oracle.decode_attn(case.q_lat, case.q_pe, case.pool, case.page_table,
                                case.seq_lens, case.scale, lib=lib)
    o2, l2 = oracle.decode_attn(case.q_lat.double(), case.q_pe.double(), case.pool.double(),
                                case.page_table, case.seq_lens, case.scale, lib=lib)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def pin_weight_spread(lib):
    """The rounding sensitivity D = sum_j a_j |c_j - o| (test infrastructure):
    0 for one cached row and for equal rows; for q = 0 (uniform weights) the
    mean absolute deviation about the mean (numpy); and the largest change of
    o under weight errors of at most u, found by perturbing the weights
    directly, is u D to first order (reached by e_j = u sign(c_j - o))."""
    case = _small_case(lens=(1, 50, 64), seed=31)
    d_c = case.q_lat.shape[3]
    args = (case.q_lat, case.q_pe, case.pool, case.page_table, case.seq_lens, case.scale)
    D = oracle.weight_spread(*args, lib=lib)
    o, _ = oracle.decode_attn(*args, lib=lib)
    assert np.abs(D[0]).max() < 1e-14  # a single row: o = c_0
    u = 2.0 ** -8
    g = np.random.default_rng(3)
    for b, i in [(1, 0), (2, 3)]:
        rows = _gather_kv(case, b)[:, :d_c].numpy()
        a = oracle.attention_weights(*args[:5], case.scale, b, 0, i, lib=lib)
        for _ in range(3):  # random errors stay within u / (1 - u) D
            e = g.uniform(-u, u, a.shape)
            w = a * (1 + e)
            o2 = (w / w.sum()) @ rows
            assert (np.abs(o2 - o[b, 0, i]) <= u / (1 - u) * D[b, 0, i] + 1e-12).all()
        for c in (0, d_c // 2, d_c - 1):  # the worst sign pattern reaches u D / (1 + ebar)
            e = u * np.sign(rows[:, c] - o[b, 0, i, c])
            w = a * (1 + e)
            moved = abs(((w / w.sum()) @ rows[:, c]) - o[b, 0, i, c])
            assert abs(moved * (1 + (a * e).sum()) - u * D[b, 0, i, c]) <= 1e-12 * (1 + D[b, 0, i, c])
    zero = _small_case(lens=(1, 50, 64), seed=31)
    zero.q_lat.zero_()
    zero.q_pe.zero_()
    Dz = oracle.weight_spread(zero.q_lat, zero.q_pe, zero.pool, zero.page_table, zero.seq_lens,
                              zero.scale, lib=lib)
    for b in (1, 2):
        rows = _gather_kv(zero, b)[:, :d_c].numpy()
        mad = np.abs(rows - rows.mean(0)).mean(0)
        assert np.abs(Dz[b, 0] - mad).max() < 1e-13
    same = _small_case(lens=(5, 40, 64), seed=32)
    same.pool[:] = same.pool[0, 0]
    Ds = oracle.weight_spread(same.q_lat, same.q_pe, same.pool, same.page_table, same.seq_lens,
                              same.scale, lib=lib)
    assert np.abs(Ds).max() < 1e-13


def pin_naive_prefill(lib):
    """Training-form attention with every token a query: equal to the naive
    route with T = L causal queries, and to torch's fp64 causal
    scaled_dot_product_attention on keys and values expanded by matmul
    ([Mishra] "Multi-head Latent Attention": the unabsorbed form); a
    selection of rows equals those rows of the full result."""
    g = torch.Generator().manual_seed(41)
    B, L, H, d_h, d_c, d_r = 2, 37, 3, 8, 16, 4
    cache = torch.randn((B, L, d_c + d_r), generator=g, dtype=torch.float64)
    qn = torch.randn((B, L, H, d_h), generator=g, dtype=torch.float64)
    qp = torch.randn((B, L, H, d_r), generator=g, dtype=torch.float64)
    w_uk = torch.randn((H, d_h, d_c), generator=g, dtype=torch.float64) / 4
    w_uv = torch.randn((H, d_h, d_c), generator=g, dtype=torch.float64) / 4
    scale = 1.0 / math.sqrt(d_h + d_r)
    u, lse = oracle.naive_prefill(cache.numpy(), qn, qp, w_uk, w_uv, scale, causal=True, lib=lib)
    u_dec, _ = oracle.naive_decode(cache.reshape(B * L, -1).numpy(), qn, qp, w_uk, w_uv, None, L,
                                   scale, causal=True, lib=lib)
    assert np.abs(u - u_dec).max() < 1e-12
    c = cache[..., :d_c]
    k = torch.cat([torch.einsum("blc,hec->bhle", c, w_uk),
                   cache[..., d_c:].unsqueeze(1).expand(B, H, L, d_r)], -1)
    v = torch.einsum("blc,hec->bhle", c, w_uv)
    q = torch.cat([qn, qp], -1).permute(0, 2, 1, 3)
    for causal in (True, False):
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)
        got, lse_c = oracle.naive_prefill(cache.numpy(), qn, qp, w_uk, w_uv, scale, causal=causal,
                                          lib=lib)
        assert np.abs(got - ref.permute(0, 2, 1, 3).numpy()).max() < 1e-12
        s = (q @ k.transpose(-1, -2)) * scale
        if causal:
            s = s.masked_fill(torch.ones(L, L, dtype=torch.bool).triu(1), float("-inf"))
        assert np.abs(lse_c - torch.logsumexp(s, -1).permute(0, 2, 1).numpy()).max() < 1e-12
    sel = np.array([0, 5, B * L * H - 1, 100])
    us, ls = oracle.naive_prefill(cache.numpy(), qn, qp, w_uk, w_uv, scale, causal=True, sel=sel,
                                  lib=lib)
    assert np.array_equal(us, u.reshape(-1, d_h)[sel]) and np.array_equal(ls, lse.reshape(-1)[sel])


def pin_prefill_attn(lib):
    """Attention of given keys and values equals the training-form route on
    the exact expansions of the same cache (so it is the route's attention
    half), and torch's fp64 causal scaled_dot_product_attention; the RoPE key
    may be read from cache rows at a column offset."""
    g = torch.Generator().manual_seed(43)
    B, L, H, d_h, d_c, d_r = 2, 29, 3, 8, 16, 4
    cache = torch.randn((B, L, d_c + d_r), generator=g, dtype=torch.float64)
    qn = torch.randn((B * L, H, d_h), generator=g, dtype=torch.float64)
    qp = torch.randn((B * L, H, d_r), generator=g, dtype=torch.float64)
    w_uk = torch.randn((H, d_h, d_c), generator=g, dtype=torch.float64) / 4
    w_uv = torch.randn((H, d_h, d_c), generator=g, dtype=torch.float64) / 4
    scale = 1.0 / math.sqrt(d_h + d_r)
    c = cache.reshape(B * L, -1)[:, :d_c]
    kn = torch.einsum("rc,hec->rhe", c, w_uk)
    vv = torch.einsum("rc,hec->rhe", c, w_uv)
    rows = cache.reshape(B * L, -1)
    u, lse = oracle.prefill_attn(qn, qp, kn, rows, vv, L, scale, causal=True, k_pe_off=d_c, lib=lib)
    u_ref, lse_ref = oracle.naive_prefill(cache.numpy(), qn.reshape(B, L, H, d_h),
                                          qp.reshape(B, L, H, d_r), w_uk, w_uv, scale, lib=lib)
    assert np.abs(u - u_ref.reshape(u.shape)).max() < 1e-12
    assert np.abs(lse - lse_ref.reshape(lse.shape)).max() < 1e-12
    q = torch.cat([qn, qp], -1).reshape(B, L, H, -1).permute(0, 2, 1, 3)
    k = torch.cat([kn, rows[:, d_c:].unsqueeze(1).expand(B * L, H, d_r)], -1)
    k = k.reshape(B, L, H, -1).permute(0, 2, 1, 3)
    v = vv.reshape(B, L, H, d_h).permute(0, 2, 1, 3)
    for causal in (True, False):
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)
        got, _ = oracle.prefill_attn(qn, qp, kn, rows, vv, L, scale, causal=causal, k_pe_off=d_c,
                                     lib=lib)
        assert np.abs(got - ref.permute(0, 2, 1, 3).reshape(B * L, H, d_h).numpy()).max() < 1e-12


ALL_PINS = [
    pin_cache_accounting, pin_absorption_cost, pin_rope, pin_naive_equals_absorbed,
    pin_naive_equals_absorbed_at_model_widths, pin_naive_vs_library_sdpa, pin_project_vs_library, pin_position_shift_invariance,
    pin_decode_vs_library_sdpa, pin_decode_closed_forms, pin_softmax_rows_sum_to_one,
    pin_fp64_rounding_is_negligible, pin_page_permutation_invariance, pin_combine_split_identity, pin_empty_sequence,
    pin_out_proj_vs_library, pin_bf16_widening, pin_weight_spread, pin_naive_prefill,
    pin_prefill_attn,
]
