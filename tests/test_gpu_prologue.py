"""The cache write and the query projection (mla_cache_append,
mla_project_q) against the fp64 oracle (needs a B300).

Each token's cache row [c ; k^R] = [W^DKV h ; RoPE(W^KR h, pos)] and query
[q^C ; q^R] per head (q^R rotated at pos) come from the oracle's projection
of the token as a one-position sequence (position 0, where RoPE is the
identity), rotated at the token's own position by the oracle's RoPE.
Tolerances:
    fp32 mode: max abs error <= 1e-4 (the decode's fp32 bar).
    bf16 mode: |x - x*| <= 2^-8 |x*| + 1e-5 elementwise: one rounding to
        bf16 (half a unit in the last place; bf16 keeps 8 significant bits,
        so at most 2^-8 |x*|) of an fp32 accumulation whose own error is
        orders of magnitude smaller.  The query's RoPE part is rounded twice:
        the GEMM's bf16 output (a pair's input error is then at most 2^-8 of
        the pair's norm, and a rotation keeps norms) and the rotated value
        (2^-8 |y|), so there the bar is 2^-7 of the pair's norm.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_71_b300 import mla, workloads

pytestmark = pytest.mark.gpu

FP32_MAX = 1e-4
BF16_REL, BF16_ABS = 2.0 ** -8, 1e-5


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.library()
    yield


@pytest.fixture(autouse=True)
def _device_status():
    """Each test starts with a clear device status word and must leave it clear."""
    mla.get_device_status()
    yield
    code, detail = mla.get_device_status()
    assert code == 0, f"device status {code}: site {detail & 0xFFF:#x}"


def _oracle_kv_rows(h, w_dkv, w_kr, positions):
    """[c ; RoPE(k^R, pos)] of every token (rows of h), from the oracle."""
    N, d = h.shape
    d_r = w_kr.shape[0]
    w_q = torch.zeros((2 + d_r, d), dtype=h.dtype)  # one 2-wide head: the query is unused here
    rows, _, _ = oracle.project(h.cpu().reshape(N, 1, d), w_dkv.cpu(), w_kr.cpu(), w_q, 1, 2, qpos=0)
    d_c = w_dkv.shape[0]
    for n, pos in enumerate(positions.tolist()):
        rows[n, d_c:] = oracle.rope(rows[n, d_c:], pos)
    return rows


def _oracle_query(h, w_q, positions, H, d_h, d_r):
    """(q^C [N,H,d_h], RoPE(q^R, pos) [N,H,d_r]) of every token, from the oracle."""
    N, d = h.shape
    w_dkv = torch.zeros((2, d), dtype=h.dtype)
    w_kr = torch.zeros((d_r, d), dtype=h.dtype)
    _, qn, qp = oracle.project(h.cpu().reshape(N, 1, d), w_dkv, w_kr, w_q.cpu(), H, d_h, qpos=0)
    for n, pos in enumerate(positions.tolist()):
        for i in range(H):
            qp[n, i] = oracle.rope(qp[n, i], pos)
    return qn, qp


def _pool_for(seqs, positions, B, page, width, dtype, seed):
    """A NaN-filled pool with one (permuted) page for every page the tokens touch."""
    max_pages = int(positions.max()) // page + 1
    used = sorted({(int(s), int(p) // page) for s, p in zip(seqs.tolist(), positions.tolist())})
    perm = torch.randperm(len(used), generator=torch.Generator().manual_seed(seed))
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    for k, (s, lp) in enumerate(used):
        table[s, lp] = int(perm[k])
    pool = torch.full((len(used), page, width), float("nan"), dtype=dtype)
    return pool, table


def _rows_of(pool, table, seqs, positions):
    page = pool.shape[1]
    pg = table[seqs.long(), (positions // page).long()].long()
    return pool[pg, (positions % page).long()]


def _untouched(pool, table, seqs, positions):
    """Every pool row the tokens do not name still holds its NaN fill."""
    page = pool.shape[1]
    mask = torch.ones(pool.shape[:2], dtype=torch.bool)
    pg = table[seqs.long(), (positions // page).long()].long()
    mask[pg, (positions % page).long()] = False
    return bool(torch.isnan(pool[mask].float()).all())


def _bf16_close(got, ref):
    got = np.asarray(got.float().cpu(), dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64).reshape(got.shape)
    excess = (np.abs(got - ref) - (BF16_REL * np.abs(ref) + BF16_ABS)).max()
    return excess <= 0, float(np.abs(got - ref).max())


def test_fp32_tiny_model_fully_on_the_gpu():
    """The tiny fp32 model from hidden states to the layer output, every step
    on the GPU: cache write of all 2 x 128 positions (in shuffled order),
    query of the last token, absorb, decode, output projection; against the
    oracle's naive route (K and V expanded)."""
    m = workloads.tiny_model(seed=0)
    B, L, H, d_h, d_c, d_r, d = m["B"], m["L"], m["H"], m["d_h"], m["d_c"], m["d_r"], m["d"]
    cache, q_nope_ref, q_pe_ref = oracle.project(m["h"].double(), m["w_dkv"], m["w_kr"], m["w_q"],
                                                 H, d_h, qpos=L - 1)
    _, out_ref = oracle.naive_decode(cache, q_nope_ref[:, None], q_pe_ref[:, None], m["w_uk"],
                                     m["w_uv"], m["w_o"], L, m["scale"])
    dev = "cuda"
    h = m["h"].reshape(B * L, d)
    order = torch.randperm(B * L, generator=torch.Generator().manual_seed(1))
    seqs = (torch.arange(B * L) // L).to(torch.int32)[order]
    positions = (torch.arange(B * L) % L).to(torch.int32)[order]
    pool, table = _pool_for(seqs, positions, B, 64, d_c + d_r, torch.float32, seed=2)
    pool_d, table_d = pool.to(dev), table.to(dev)
    mla.cache_append(h[order].contiguous().to(dev), m["w_dkv"].to(dev), m["w_kr"].to(dev),
                     seqs.to(dev), positions.to(dev), table_d, pool_d)
    last = torch.arange(B) * L + (L - 1)
    qpos = torch.full((B,), L - 1, dtype=torch.int32)
    qn, qp = mla.project_q(h[last].contiguous().to(dev), m["w_q"].to(dev), qpos.to(dev), H, d_h, d_r)
    q_lat = mla.absorb_q(qn, m["w_uk"].to(dev))
    o, lse = mla.decode_attn(q_lat.view(B, 1, H, d_c), qp.view(B, 1, H, d_r), pool_d, table_d,
                             torch.full((B,), L, dtype=torch.int32, device=dev), m["scale"])
    out = mla.out_proj(o.view(B, H, d_c), m["w_uv"].to(dev), m["w_o"].to(dev))
    torch.cuda.synchronize()
    rows = _rows_of(pool_d.cpu(), table, torch.arange(B * L) // L, torch.arange(B * L) % L)
    assert np.abs(rows.double().numpy() - cache).max() <= FP32_MAX
    assert np.abs(qn.cpu().double().numpy() - q_nope_ref).max() <= FP32_MAX
    assert np.abs(qp.cpu().double().numpy() - q_pe_ref).max() <= FP32_MAX
    assert np.abs(out.cpu().double().numpy() - out_ref.reshape(B, d)).max() <= FP32_MAX


def test_fp32_odd_widths():
    """fp32 widths whose 8-row tiles straddle W^DKV / W^KR and the heads of
    W^Q (d_c = 60, d_r = 10; heads of 6 + 4 rows), ragged token count."""
    N, d, d_c, d_r, B, page, H, d_h = 13, 100, 60, 10, 3, 16, 3, 6
    g = torch.Generator().manual_seed(11)
    h = torch.randn((N, d), generator=g)
    w_dkv = workloads.weight((d_c, d), d, g, "cpu", torch.float32)
    w_kr = workloads.weight((d_r, d), d, g, "cpu", torch.float32)
    w_q = workloads.weight((H * (d_h + d_r), d), d, g, "cpu", torch.float32)
    seqs = torch.randint(0, B, (N,), generator=g, dtype=torch.int32)
    positions = torch.randperm(500, generator=g)[:N].to(torch.int32)  # distinct: no shared row
    pool, table = _pool_for(seqs, positions, B, page, d_c + d_r, torch.float32, seed=12)
    pool_d = pool.cuda()
    mla.cache_append(h.cuda(), w_dkv.cuda(), w_kr.cuda(), seqs.cuda(), positions.cuda(),
                     table.cuda(), pool_d)
    qn, qp = mla.project_q(h.cuda(), w_q.cuda(), positions.cuda(), H, d_h, d_r)
    torch.cuda.synchronize()
    got = _rows_of(pool_d.cpu(), table, seqs, positions)
    ref = _oracle_kv_rows(h, w_dkv, w_kr, positions)
    assert np.abs(got.double().numpy() - ref).max() <= FP32_MAX
    assert _untouched(pool_d.cpu(), table, seqs, positions)
    qn_ref, qp_ref = _oracle_query(h, w_q, positions, H, d_h, d_r)
    assert np.abs(qn.cpu().double().numpy() - qn_ref).max() <= FP32_MAX
    assert np.abs(qp.cpu().double().numpy() - qp_ref).max() <= FP32_MAX


def _kv_tokens(N, B, g):
    """N distinct (sequence, position) pairs: two pairs of neighbours in one
    page, the rest spread up to position 131071."""
    pairs = {(0, 5), (0, 6), (1, 64), (1, 127)}
    while len(pairs) < N:
        pairs.add((int(torch.randint(0, B, (1,), generator=g)),
                   int(torch.randint(0, 131072, (1,), generator=g))))
    pairs = sorted(pairs, key=lambda p: torch.rand(1, generator=g).item())
    seqs = torch.tensor([p[0] for p in pairs], dtype=torch.int32)
    positions = torch.tensor([p[1] for p in pairs], dtype=torch.int32)
    return seqs, positions


@pytest.mark.parametrize("N", [37, 300])
def test_bf16_cache_append_model_widths(N):
    """d = 7168 -> [c 512 ; k^R 64], tokens at scattered positions up to
    131071 (several 8-token tiles and a ragged tail; 300 tokens take two
    GEMM column tiles)."""
    d, d_c, d_r, B = 7168, 512, 64, 5
    g = torch.Generator().manual_seed(40 + N)
    h = torch.randn((N, d), generator=g).to(torch.bfloat16)
    w_dkv = workloads.weight((d_c, d), d, g, "cpu", torch.bfloat16)
    w_kr = workloads.weight((d_r, d), d, g, "cpu", torch.bfloat16)
    seqs, positions = _kv_tokens(N, B, g)
    pool, table = _pool_for(seqs, positions, B, 64, d_c + d_r, torch.bfloat16, seed=N)
    pool_d = pool.cuda()
    mla.cache_append(h.cuda(), w_dkv.cuda(), w_kr.cuda(), seqs.cuda(), positions.cuda(),
                     table.cuda(), pool_d)
    torch.cuda.synchronize()
    got = _rows_of(pool_d.cpu(), table, seqs, positions)
    ref = _oracle_kv_rows(h, w_dkv, w_kr, positions)
    ok, err = _bf16_close(got, ref)
    assert ok, f"max |row - row*| = {err:.3e}"
    assert np.abs(ref).max() > 1.0  # not a vacuous zero
    assert _untouched(pool_d.cpu(), table, seqs, positions)


@pytest.mark.parametrize("N,d,H,d_h,d_r", [
    (19, 1536, 128, 128, 64),   # c^Q -> 128 x [128 ; 64]: the GEMM writes the heads (one N tile)
    (64, 1536, 128, 128, 64),   # the decode batch of the headline workload
    (300, 1024, 32, 128, 64),   # two N tiles, the second ragged
    (37, 1024, 128, 64, 32),    # heads of 96 rows straddle the GEMM's 128-row tiles
    (23, 1536, 8, 128, 64),     # few heads: K split into partials, then the finishing kernel
])
def test_bf16_project_q_widths(N, d, H, d_h, d_r):
    """The query projection at model widths, positions up to 10^5, against
    the oracle: content part within the bf16 bar, RoPE part within it
    relative to the length of each rotated pair."""
    g = torch.Generator().manual_seed(50 + N)
    h = torch.randn((N, d), generator=g).to(torch.bfloat16)
    w_q = workloads.weight((H * (d_h + d_r), d), d, g, "cpu", torch.bfloat16)
    positions = torch.randint(0, 100001, (N,), generator=g, dtype=torch.int32)
    qn = torch.full((N, H, d_h), float("nan"), dtype=torch.bfloat16, device="cuda")
    qp = torch.full((N, H, d_r), float("nan"), dtype=torch.bfloat16, device="cuda")
    mla.project_q(h.cuda(), w_q.cuda(), positions.cuda(), H, d_h, d_r, qn, qp)
    torch.cuda.synchronize()
    assert mla.get_device_status()[0] == 0
    qn_ref, qp_ref = _oracle_query(h, w_q, positions, H, d_h, d_r)
    ok, err = _bf16_close(qn, qn_ref)
    assert ok, f"max |q^C - q^C*| = {err:.3e}"
    got = qp.float().cpu().double().numpy()
    assert np.isfinite(got).all()
    pair = np.sqrt(qp_ref[..., 0::2] ** 2 + qp_ref[..., 1::2] ** 2).repeat(2, axis=-1)
    excess = (np.abs(got - qp_ref) - (2 * BF16_REL * pair + BF16_ABS)).max()
    assert excess <= 0, f"max |q^R - q^R*| = {np.abs(got - qp_ref).max():.3e}"


def test_cache_append_bad_page_raises_device_status():
    """A token whose page-table entry is missing raises the status word and
    writes nothing outside the tokens' rows; the context stays usable and the
    next call with a valid table writes every row."""
    N, d, d_c, d_r, B = 9, 512, 128, 64, 2
    g = torch.Generator().manual_seed(60)
    h = torch.randn((N, d), generator=g).to(torch.bfloat16)
    w_dkv = workloads.weight((d_c, d), d, g, "cpu", torch.bfloat16)
    w_kr = workloads.weight((d_r, d), d, g, "cpu", torch.bfloat16)
    seqs = torch.tensor([0, 0, 1, 1, 0, 1, 0, 1, 1], dtype=torch.int32)
    positions = torch.tensor([0, 1, 2, 3, 64, 65, 130, 131, 200], dtype=torch.int32)
    pool, table = _pool_for(seqs, positions, B, 64, d_c + d_r, torch.bfloat16, seed=61)
    bad = table.clone()
    bad[1, 200 // 64] = -1  # the last token's page
    pool_d = pool.cuda()
    mla.cache_append(h.cuda(), w_dkv.cuda(), w_kr.cuda(), seqs.cuda(), positions.cuda(),
                     bad.cuda(), pool_d)
    code, _ = mla.get_device_status()
    assert code == 5
    assert _untouched(pool_d.cpu(), table, seqs, positions)
    assert torch.isnan(_rows_of(pool_d.cpu(), table, seqs[8:], positions[8:]).float()).all()
    mla.cache_append(h.cuda(), w_dkv.cuda(), w_kr.cuda(), seqs.cuda(), positions.cuda(),
                     table.cuda(), pool_d)
    torch.cuda.synchronize()
    assert mla.get_device_status()[0] == 0
    ok, err = _bf16_close(_rows_of(pool_d.cpu(), table, seqs, positions),
                          _oracle_kv_rows(h, w_dkv, w_kr, positions))
    assert ok, f"max |row - row*| = {err:.3e}"
