"""CUDA path vs the fp64 oracle on identical seeded inputs (needs a B300).

Every call goes through the C ABI (``mla_latent_kv_71_b300.mla``).
Tolerances (bf16 storage, fp32 accumulation; ``tests/bars.py``):
    o   : |o - o*| <= 2e-2 elementwise where |o|, |o*| < 8, plus half a bf16
          spacing where the larger of the two is >= 8 (only there does the
          rounding to bf16 alone reach 2e-2), and
          ||o - o*||_F / ||o*||_F <= 5e-3 over the whole tensor
    lse : max |lse - lse*| <= 1e-3
    fp32 mode: max abs error <= 1e-4 on o, lse and out.
The same bars apply to the final projection output of the end-to-end cases.
The full-size workloads are compared element by element on every row.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_71_b300 import mla, workloads
from tests.bars import FP32_MAX, LSE_MAX, O_FRO, O_MAX, o_bar, o_excess

pytestmark = pytest.mark.gpu


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
    assert code == 0, f"device status {code}: site {detail & 0xFFF:#x} block {detail >> 12}"


def _to(case: workloads.DecodeCase, device):
    return workloads.DecodeCase(case.q_lat.to(device), case.q_pe.to(device), case.pool.to(device),
                                case.page_table.to(device), case.seq_lens.to(device), case.scale,
                                case.causal, dict(case.extra))


def _spread_fn(case):
    """Weight spread of listed flattened (b, t, head) rows of a decode case."""
    c = _to(case, "cpu")
    return lambda rows: oracle.weight_spread(c.q_lat, c.q_pe, c.pool, c.page_table, c.seq_lens,
                                             c.scale, causal=c.causal, sel=rows)


def _check_o_lse(o, lse, o_ref, lse_ref, what="", case=None):
    o = np.asarray(o.float().cpu() if isinstance(o, torch.Tensor) else o, dtype=np.float64)
    lse = np.asarray(lse.float().cpu() if isinstance(lse, torch.Tensor) else lse, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64).reshape(o.shape)
    lse_ref = np.asarray(lse_ref, dtype=np.float64).reshape(lse.shape)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: lse finiteness differs"
    assert np.isfinite(o).all(), f"{what}: non-finite o"
    err, excess, err_small, n_spread = o_excess(o, o_ref, _spread_fn(case) if case else None)
    fro = np.linalg.norm(o - o_ref) / max(np.linalg.norm(o_ref), 1e-30)
    lerr = np.abs(lse[fin] - lse_ref[fin]).max() if fin.any() else 0.0
    print(f"[parity] {what}: max|o-o*| {err:.3e} (on |o*|<8: {err_small:.3e} vs {O_MAX}), "
          f"rel fro {fro:.3e}, max|lse-lse*| {lerr:.3e}, rows {o.size // o.shape[-1]}, "
          f"rows under the weight-rounding bound {n_spread}")
    assert excess <= 0, f"{what}: max |o - o*| = {err:.3e} exceeds the bar by {excess:.3e}"
    assert fro <= O_FRO, f"{what}: rel Frobenius = {fro:.3e}"
    assert lerr <= LSE_MAX, f"{what}: max |lse - lse*| = {lerr:.3e}"
    return err, fro, lerr


def _run_decode(case, **kw):
    torch.cuda.synchronize()
    o, lse = mla.decode_attn(case.q_lat, case.q_pe, case.pool, case.page_table, case.seq_lens,
                             case.scale, causal=case.causal, **kw)
    torch.cuda.synchronize()
    return o, lse


def _oracle_decode(case, sel=None):
    c = _to(case, "cpu")
    return oracle.decode_attn(c.q_lat, c.q_pe, c.pool, c.page_table, c.seq_lens, c.scale,
                              causal=c.causal, sel=sel)


# ------------------------------------------------------------ fp32 mode

def test_fp32_decode_tiny_shapes():
    spec = workloads.WORKLOADS["tiny_fp32"]
    case = workloads.decode_case(2, 1, spec["H"], spec["d_c"], spec["d_r"], spec["lens"],
                                 seed=0, dtype=torch.float32, device="cuda", d_h=spec["d_h"])
    o, lse = _run_decode(case)
    o_ref, lse_ref = _oracle_decode(case)
    assert np.abs(o.cpu().double().numpy() - o_ref).max() <= FP32_MAX
    assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= FP32_MAX


def test_fp32_end_to_end_tiny_widths():
    """absorb_q -> decode -> out_proj in fp32 at the tiny model's widths."""
    B, H, d_h, d_c, d_r, d = 2, 8, 32, 64, 16, 256
    case = workloads.decode_case(B, 1, H, d_c, d_r, [128, 77], page=16, seed=3,
                                 dtype=torch.float32, device="cuda", d_h=d_h)
    qn = workloads.q_nope(B, 1, H, d_h, seed=4, device="cuda", dtype=torch.float32)
    w_uk, w_uv, w_o = workloads.projection_weights(H, d_h, d_c, d, seed=5, device="cuda",
                                                   dtype=torch.float32)
    q_lat = mla.absorb_q(qn.view(B, H, d_h), w_uk)
    o, lse = mla.decode_attn(q_lat.view(B, 1, H, d_c), case.q_pe, case.pool, case.page_table,
                             case.seq_lens, case.scale)
    out = mla.out_proj(o.view(B, H, d_c), w_uv, w_o)
    torch.cuda.synchronize()
    cpu = _to(case, "cpu")
    q_ref = oracle.absorb_q(qn.cpu().view(B, H, d_h), w_uk.cpu())
    o_ref, lse_ref = oracle.decode_attn(q_ref.reshape(B, 1, H, d_c), cpu.q_pe, cpu.pool,
                                        cpu.page_table, cpu.seq_lens, cpu.scale)
    out_ref, _ = oracle.out_proj(o_ref.reshape(B, H, d_c), w_uv.cpu(), w_o.cpu())
    assert np.abs(q_lat.cpu().double().numpy() - q_ref).max() <= FP32_MAX
    assert np.abs(o.cpu().double().numpy() - o_ref).max() <= FP32_MAX
    assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= FP32_MAX
    assert np.abs(out.cpu().double().numpy() - out_ref).max() <= FP32_MAX


# ------------------------------------------------------------ bf16 decode

SMALL = [
    # (B, T, H, lens) -- several pages, ragged tails, a 1-token sequence
    (3, 1, 128, [1, 65, 200]),
    (4, 1, 128, [64, 128, 640, 1000]),
    (2, 2, 128, [2, 129]),          # two causal query tokens
    (3, 1, 16, [33, 64, 300]),      # fewer heads than the tile
    (2, 1, 200, [70, 130]),         # two head groups
    (2, 3, 128, [3, 250]),          # three causal query tokens
]


@pytest.mark.parametrize("B,T,H,lens", SMALL, ids=[f"B{c[0]}T{c[1]}H{c[2]}" for c in SMALL])
def test_bf16_decode_small(B, T, H, lens):
    case = workloads.decode_case(B, T, H, 512, 64, lens, seed=11 + B + T + H, device="cuda")
    o, lse = _run_decode(case)
    o_ref, lse_ref = _oracle_decode(case)
    _check_o_lse(o, lse, o_ref, lse_ref, f"B{B}T{T}H{H}", case)


def test_bf16_decode_many_sequences_split_across_clusters():
    """More pages than clusters: most sequences are cut between SMs and merged."""
    lens = [int(x) for x in torch.randint(1, 3000, (24,), generator=torch.Generator().manual_seed(5))]
    case = workloads.decode_case(24, 1, 128, 512, 64, lens, seed=21, device="cuda")
    o, lse = _run_decode(case)
    o_ref, lse_ref = _oracle_decode(case)
    _check_o_lse(o, lse, o_ref, lse_ref, "many", case)
    o2, lse2 = _run_decode(case, seq_lens_host=case.seq_lens.cpu())
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_bf16_decode_empty_sequence():
    case = workloads.decode_case(3, 1, 128, 512, 64, [0, 70, 5], seed=22, device="cuda")
    o, lse = _run_decode(case)
    assert torch.isneginf(lse[0]).all() and (o[0] == 0).all()
    o_ref, lse_ref = _oracle_decode(case)
    _check_o_lse(o, lse, o_ref, lse_ref, "empty", case)


def test_bf16_decode_ignores_nan_past_the_end():
    """Rows past a sequence's length may hold NaN: they must not reach o."""
    case = workloads.decode_case(2, 1, 128, 512, 64, [70, 5], seed=23, device="cuda")
    o_ref, lse_ref = _oracle_decode(case)
    page = case.pool.shape[1]
    for b, n in enumerate([70, 5]):
        last = int(case.page_table[b, (n - 1) // page])
        case.pool[last, n % page:] = float("nan")
    o, lse = _run_decode(case)
    _check_o_lse(o, lse, o_ref, lse_ref, "nan-tail")


def test_bf16_decode_page_permutation_is_bitwise_invariant():
    case = workloads.decode_case(3, 1, 128, 512, 64, [100, 700, 64], seed=24, device="cuda")
    o1, l1 = _run_decode(case)
    P = case.pool.shape[0]
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(9))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P)
    pool2 = case.pool[perm.cuda()].contiguous()
    table2 = case.page_table.clone()
    valid = table2 >= 0
    table2[valid] = inv.cuda()[table2[valid].long()].to(torch.int32)
    o2, l2 = mla.decode_attn(case.q_lat, case.q_pe, pool2, table2, case.seq_lens, case.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_bf16_decode_head_order_equivariance():
    case = workloads.decode_case(2, 1, 128, 512, 64, [300, 90], seed=25, device="cuda")
    o1, l1 = _run_decode(case)
    perm = torch.randperm(128, generator=torch.Generator().manual_seed(2)).cuda()
    o2, l2 = mla.decode_attn(case.q_lat[:, :, perm].contiguous(), case.q_pe[:, :, perm].contiguous(),
                             case.pool, case.page_table, case.seq_lens, case.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1[:, :, perm], o2) and torch.equal(l1[:, :, perm], l2)


def test_bf16_decode_hot_rows_stress_rescaling():
    """A few latent rows scaled by 8 make the running maximum jump late."""
    case = workloads.decode_case(2, 1, 128, 512, 64, [2000, 900], seed=26, device="cuda",
                                 hot_frac=0.01)
    o, lse = _run_decode(case)
    o_ref, lse_ref = _oracle_decode(case)
    _check_o_lse(o, lse, o_ref, lse_ref, "hot", case)


def test_bf16_decode_bad_page_id_raises_device_status():
    case = workloads.decode_case(2, 1, 128, 512, 64, [100, 100], seed=27, device="cuda")
    case.page_table[1, 0] = case.pool.shape[0] + 5
    _run_decode(case)
    code, _ = mla.get_device_status()
    assert code == 5
    case.page_table[1, 0] = 0
    o, lse = _run_decode(case)  # the context is still usable
    assert mla.get_device_status()[0] == 0
    assert torch.isfinite(lse).all()


# ----------------------------------------------------- combine, projections

def test_combine_splits_matches_oracle():
    g = torch.Generator(device="cuda").manual_seed(31)
    S, rows, d_c = 3, 300, 512
    o_part = torch.randn((S, rows, d_c), generator=g, device="cuda")
    lse_part = torch.randn((S, rows), generator=g, device="cuda") * 3
    lse_part[1, :10] = float("-inf")
    lse_part[:, 20] = float("-inf")
    for dt in (torch.float32, torch.bfloat16):
        o, lse = mla.combine_splits(o_part, lse_part, out_dtype=dt)
        torch.cuda.synchronize()
        o_ref, lse_ref = oracle.combine(o_part.cpu().numpy(), lse_part.cpu().numpy())
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(lse.cpu().numpy()), fin)
        tol = FP32_MAX if dt == torch.float32 else O_MAX
        assert np.abs(o.float().cpu().numpy() - o_ref).max() <= tol
        assert np.abs(lse.cpu().numpy()[fin] - lse_ref[fin]).max() <= 1e-4


@pytest.mark.parametrize("rows,H", [(64, 128), (64, 16), (5, 8), (300, 2)])
def test_bf16_absorb_q(rows, H):
    qn = workloads.q_nope(rows, 1, H, 128, seed=41, device="cuda").view(rows, H, 128)
    w_uk, _, _ = workloads.projection_weights(H, 128, 512, 128, seed=42, device="cuda")
    q_lat = mla.absorb_q(qn, w_uk)
    torch.cuda.synchronize()
    ref = oracle.absorb_q(qn.cpu(), w_uk.cpu())
    got = q_lat.float().cpu().numpy()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= O_FRO and (np.abs(got - ref) <= o_bar(got, ref)).all()


@pytest.mark.parametrize("rows,H,d", [(64, 128, 7168), (64, 16, 7168), (7, 4, 256)])
def test_bf16_out_proj(rows, H, d):
    g = torch.Generator(device="cuda").manual_seed(43)
    o = (torch.randn((rows, H, 512), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    _, w_uv, w_o = workloads.projection_weights(H, 128, 512, d, seed=44, device="cuda")
    out = mla.out_proj(o, w_uv, w_o)
    out2 = mla.out_proj(o, w_uv, w_o)  # counters of the split-K reduction are reusable
    torch.cuda.synchronize()
    ref, _ = oracle.out_proj(o.cpu(), w_uv.cpu(), w_o.cpu())
    got = out.float().cpu().numpy()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= O_FRO, rel
    assert np.abs(got - ref).max() <= O_MAX
    assert torch.equal(out, out2)


# ------------------------------------------ full-size workloads (every row)

@pytest.mark.parametrize("name", ["decode_b64_h128_l4096", "ragged_b128_l16k", "long_b4_l128k"])
def test_full_size_workloads_every_row(name):
    """The GPU over the whole workload, in the launch configuration the bench
    times (lengths also on the host: at the headline batch that is one
    cluster per sequence, no unit cut), and without host lengths (all
    clusters, units cut and merged); the oracle on every (sequence, token,
    head) row of both."""
    case = workloads.make_workload(name, device="cuda")
    o_ref, lse_ref = _oracle_decode(case)
    for host in (True, False):
        o, lse = _run_decode(case, seq_lens_host=case.seq_lens.cpu() if host else None)
        assert torch.isfinite(lse).all() and torch.isfinite(o.float()).all()
        _check_o_lse(o, lse, o_ref, lse_ref, f"{name} ({'host lengths' if host else 'device lengths'})",
                     case)


@pytest.mark.parametrize("name", ["mtp_b32_t2_l8192", "smallhead_b64_h16_l32k"])
def test_full_size_end_to_end_every_row(name):
    """absorb_q -> decode -> out_proj at full size, every sequence compared."""
    case = workloads.make_workload(name, device="cuda")
    B, T, H, d_c = case.q_lat.shape
    qn = case.extra["q_nope"]
    w_uk, w_uv, w_o = case.extra["w_uk"], case.extra["w_uv"], case.extra["w_o"]
    q_lat = mla.absorb_q(qn.view(B * T, H, -1), w_uk).view(B, T, H, d_c)
    o, lse = mla.decode_attn(q_lat, case.q_pe, case.pool, case.page_table, case.seq_lens,
                             case.scale, causal=case.causal)
    out = mla.out_proj(o.view(B * T, H, d_c), w_uv, w_o)
    torch.cuda.synchronize()
    # Stage by stage on identical inputs: absorb from the bf16 q_nope, decode
    # from the GPU's bf16 q_lat, out_proj from the GPU's o.  Then the fp64
    # chain from q_nope, compared on the final output (q_lat and o are stored
    # in bf16 between the stages, which moves lse by up to a few 1e-3 for
    # short sequences; the chain is checked on out).
    cpu = _to(workloads.DecodeCase(q_lat, case.q_pe, case.pool, case.page_table,
                                   case.seq_lens, case.scale, case.causal), "cpu")
    q_ref = oracle.absorb_q(qn.cpu().reshape(B * T, H, -1), w_uk.cpu())
    q_got = q_lat.float().cpu().numpy().reshape(q_ref.shape)
    assert np.linalg.norm(q_got - q_ref) <= O_FRO * np.linalg.norm(q_ref)
    assert (np.abs(q_got - q_ref) <= o_bar(q_got, q_ref)).all()
    o_ref, lse_ref = oracle.decode_attn(cpu.q_lat, cpu.q_pe, cpu.pool, cpu.page_table,
                                        cpu.seq_lens, cpu.scale, causal=cpu.causal)
    _check_o_lse(o, lse, o_ref, lse_ref, name)
    w_uv_c, w_o_c = w_uv.cpu(), w_o.cpu()
    stage_ref, _ = oracle.out_proj(o.cpu().reshape(B * T, H, d_c), w_uv_c, w_o_c)
    got = out.float().cpu().numpy().reshape(stage_ref.shape)
    assert np.linalg.norm(got - stage_ref) <= O_FRO * np.linalg.norm(stage_ref)
    assert (np.abs(got - stage_ref) <= o_bar(got, stage_ref)).all()
    o64, _ = oracle.decode_attn(q_ref.reshape(B, T, H, d_c), cpu.q_pe, cpu.pool,
                                cpu.page_table, cpu.seq_lens, cpu.scale, causal=cpu.causal)
    out_ref, _ = oracle.out_proj(o64.reshape(B * T, H, d_c), w_uv_c, w_o_c)
    rel = np.linalg.norm(got - out_ref) / np.linalg.norm(out_ref)
    err, excess, _, _ = o_excess(got, out_ref)
    print(f"[parity] {name} end to end: max|out-out*| {err:.3e}, rel fro {rel:.3e}")
    assert rel <= O_FRO, rel
    assert excess <= 0, f"{name}: max |out - out*| = {err:.3e} exceeds the bar by {excess:.3e}"
