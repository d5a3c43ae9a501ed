"""Training-form prefill attention (row f3) against the fp64 oracle (needs a
B300).

The GPU path: the per-head keys and values W^UK_i c, W^UV_i c by the
tensor-core GEMM (mla_prefill_expand), causal attention with every token a
query (mla_prefill_attn), then W^O (mla_prefill_out).  Checked stage by
stage on identical inputs, as the decode path is:
  * the expansion against the oracle's per-head up-projection of the same
    latents (out_proj's first stage with o_i = c for every head): one bf16
    rounding of an fp32 sum, |x - x*| <= 2^-8 |x*| + 1e-5;
  * the attention kernel against the oracle's attention of the very bf16
    keys and values the kernel read (prefill_attn): u at the decode bars
    (|u - u*| <= 2e-2, plus half a bf16 spacing where |u| >= 8; relative
    Frobenius <= 5e-3), lse <= 1e-3;
  * u end to end against the oracle's whole route from the bf16 cache
    (naive_prefill), at the same u bars.  (Its lse is not compared end to
    end: rounding the expanded keys to bf16 moves each score by about
    scale * |q| |k| 2^-9 / sqrt(d), some 2e-3, before any attention
    arithmetic; that is the storage type's, checked in the first stage.)
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_71_b300 import mla, workloads
from tests.bars import LSE_MAX, O_FRO, o_excess

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.library()
    yield


def _gpu(case, causal=True):
    k, v = mla.prefill_expand(case.kv, case.w_uk, case.w_uv)
    u, lse = mla.prefill_attn(case.q_nope, case.q_pe, k, case.kv, v, case.L, case.scale, causal)
    torch.cuda.synchronize()
    assert mla.get_device_status()[0] == 0
    return k, v, u, lse


def _check(u, lse, u_ref, lse_ref, what):
    got = u.float().cpu().numpy().reshape(u_ref.shape)
    err, excess, _, _ = o_excess(got, u_ref)
    fro = np.linalg.norm(got - u_ref) / np.linalg.norm(u_ref)
    assert np.isfinite(got).all()
    msg = f"[parity] prefill {what}: max|u-u*| {err:.3e}, rel fro {fro:.3e}"
    if lse is not None:
        lerr = np.abs(lse.cpu().numpy().reshape(lse_ref.shape) - lse_ref).max()
        msg += f", max|lse-lse*| {lerr:.3e}"
    print(msg)
    assert excess <= 0, f"{what}: max |u - u*| = {err:.3e}"
    assert fro <= O_FRO, f"{what}: rel Frobenius {fro:.3e}"
    if lse is not None:
        assert lerr <= LSE_MAX, f"{what}: max |lse - lse*| {lerr:.3e}"


def _stages(case, k, v, u, lse, causal=True, sel=None, what=""):
    B, L = case.B, case.L
    rows, H, d_h = case.q_nope.shape
    kv = case.kv.cpu()
    d_c = kv.shape[1] - case.q_pe.shape[2]
    # 1. the expansion: W^UK_i c_r, W^UV_i c_r for every row and head
    if sel is None:
        c = kv[:, :d_c].unsqueeze(1).expand(rows, H, d_c).contiguous()
        _, k_ref = oracle.out_proj(c, case.w_uv.cpu().new_zeros((H, d_h, d_c)) + case.w_uk.cpu(),
                                   torch.zeros((128, H * d_h), dtype=torch.bfloat16))
        _, v_ref = oracle.out_proj(c, case.w_uv.cpu(), torch.zeros((128, H * d_h), dtype=torch.bfloat16))
        for got, ref in ((k, k_ref), (v, v_ref)):
            got = got.float().cpu().numpy().reshape(ref.shape)
            assert (np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5).all(), what
    # 2. attention on the kernel's own bf16 keys and values
    u_ref, lse_ref = oracle.prefill_attn(case.q_nope.cpu(), case.q_pe.cpu(), k.cpu(), kv, v.cpu(), L,
                                         case.scale, causal=causal, k_pe_off=d_c, sel=sel)
    got_u = u.reshape(-1, d_h) if sel is None else u.reshape(-1, d_h)[torch.from_numpy(sel).cuda()]
    got_l = lse.reshape(-1) if sel is None else lse.reshape(-1)[torch.from_numpy(sel).cuda()]
    _check(got_u, got_l, u_ref.reshape(-1, d_h), lse_ref.reshape(-1), what + " (attention)")
    # 3. u end to end from the bf16 cache
    cache = kv.double().numpy().reshape(B, L, -1)
    u64, _ = oracle.naive_prefill(cache, case.q_nope.cpu().reshape(B, L, H, d_h),
                                  case.q_pe.cpu().reshape(B, L, H, -1), case.w_uk.cpu(),
                                  case.w_uv.cpu(), case.scale, causal=causal, sel=sel)
    _check(got_u, None, u64.reshape(-1, d_h), None, what + " (end to end)")


@pytest.mark.parametrize("B,L,H,causal", [(2, 300, 4, True), (1, 1, 2, True), (1, 128, 3, True),
                                          (2, 129, 2, True), (2, 200, 3, False)])
def test_prefill_small(B, L, H, causal):
    case = workloads.prefill_case(B, L, H, d=256, seed=100 + L + H, device="cuda")
    k, v, u, lse = _gpu(case, causal)
    _stages(case, k, v, u, lse, causal, what=f"B{B} L{L} H{H} causal={causal}")


def test_prefill_1024_tokens_16_heads_with_out_proj():
    case = workloads.prefill_case(1, 1024, 16, d=2048, seed=110, device="cuda")
    k, v, u, lse = _gpu(case)
    out = mla.prefill_out(u, case.w_o)
    torch.cuda.synchronize()
    _stages(case, k, v, u, lse, what="L1024 H16")
    # the projection, on the GPU's own u, against the oracle's W^O product
    # (out_proj's second stage: with W^UV the identity its first is a copy)
    rows, H, d_h = u.shape
    eye = torch.eye(d_h, dtype=torch.bfloat16).repeat(H, 1, 1)  # [H, d_h, d_h]
    ref, _ = oracle.out_proj(u.cpu(), eye, case.w_o.cpu())
    got = out.float().cpu().numpy()
    _, excess, _, _ = o_excess(got, ref)
    assert excess <= 0 and np.linalg.norm(got - ref) <= O_FRO * np.linalg.norm(ref)


def test_prefill_full_size_sampled_rows():
    """4096 tokens, 128 heads (the bench's prefill workload): the oracle on
    516 sampled (position, head) rows spread over all query blocks, in the
    launch configuration the bench times."""
    case = workloads.prefill_case(1, 4096, 128, seed=111, device="cuda")
    k, v, u, lse = _gpu(case)
    H = 128
    g = np.random.default_rng(5)
    sel = np.sort(g.choice(4096 * H, size=512, replace=False))
    sel = np.unique(np.concatenate([sel, [0, H - 1, 4095 * H, 4096 * H - 1]]))
    assert torch.isfinite(u.float()).all() and torch.isfinite(lse).all()
    _stages(case, k, v, u, lse, sel=sel, what="L4096 H128 sampled")
