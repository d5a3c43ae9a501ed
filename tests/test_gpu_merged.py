"""The output projection with W^O W^UV merged ahead of time
(mla_fold_out_weights, mla_out_proj_merged) against the fp64 oracle's
unmerged out_proj (needs a B300).

Merging is an exact reassociation ([Zhang] "Value absorption: weight and
sum first, project after"), so the merged path must meet the same bars as
the unmerged one: fp32 max abs 1e-4; bf16 |out - out*| <= 2e-2 (plus half a
bf16 spacing where |out| >= 8, tests/bars.py) and relative Frobenius <= 5e-3.  (The merged weight is itself rounded to
bf16 once, which adds about one bf16 rounding to the relative error.)
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_71_b300 import mla, workloads
from tests.bars import FP32_MAX, O_FRO, o_excess

pytestmark = pytest.mark.gpu

REL = 2.0 ** -8  # one bf16 rounding, relative


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.library()
    yield


@pytest.fixture(autouse=True)
def _device_status():
    mla.get_device_status()
    yield
    code, detail = mla.get_device_status()
    assert code == 0, f"device status {code}: site {detail & 0xFFF:#x}"


def test_fp32_merged_out_proj_tiny_widths():
    rows, H, d_h, d_c, d = 5, 8, 32, 64, 256
    w_uv_, w_o_ = workloads.projection_weights(H, d_h, d_c, d, seed=70, dtype=torch.float32)[1:]
    o = torch.randn((rows, H, d_c), generator=torch.Generator().manual_seed(71))
    w_merged = mla.fold_out_weights(w_uv_.cuda(), w_o_.cuda())
    out = mla.out_proj_merged(o.cuda(), w_merged)
    torch.cuda.synchronize()
    ref, _ = oracle.out_proj(o, w_uv_, w_o_)
    assert np.abs(out.cpu().double().numpy() - ref).max() <= FP32_MAX


def test_bf16_merged_out_proj_model_widths():
    """64 rows, 16 heads of d_h 128 / d_c 512, d = 7168: the merged weight is
    7168 x 8192 (3.7x the bytes of W^UV and W^O kept apart)."""
    rows, H, d_h, d_c, d = 64, 16, 128, 512, 7168
    _, w_uv_, w_o_ = workloads.projection_weights(H, d_h, d_c, d, seed=72)
    o = torch.randn((rows, H, d_c), generator=torch.Generator().manual_seed(73)).to(torch.bfloat16)
    w_merged = mla.fold_out_weights(w_uv_.cuda(), w_o_.cuda())
    out = mla.out_proj_merged(o.cuda(), w_merged)
    torch.cuda.synchronize()
    ref, _ = oracle.out_proj(o, w_uv_, w_o_)
    got = out.float().cpu().double().numpy()
    err, excess, _, _ = o_excess(got, ref)
    fro = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert excess <= 0, f"max |out - out*| = {err:.3e}"
    assert fro <= O_FRO, f"rel Frobenius = {fro:.3e}"
    # the fold itself, on sampled entries, against the fp64 product of the
    # bf16 weights
    g = torch.Generator().manual_seed(74)
    n = torch.randint(0, d, (64,), generator=g).tolist()
    i = torch.randint(0, H, (64,), generator=g).tolist()
    c = torch.randint(0, d_c, (64,), generator=g).tolist()
    wm = w_merged.cpu().double()
    for nk, ik, ck in zip(n, i, c):
        exact = float((w_o_[nk, ik * d_h:(ik + 1) * d_h].double() * w_uv_[ik, :, ck].double()).sum())
        assert abs(float(wm[nk, ik * d_c + ck]) - exact) <= REL * abs(exact) + 1e-6


# ------------------------------------------------ query side: W^UK^T W^UQ

def _unmerged_q_lat(c_q, w_q, w_uk, H, d_h, d_r):
    """The oracle's unmerged chain: q^C_i = W^UQ_i c^Q (the content rows of
    W^Q), then q_lat_i = W^UK_i^T q^C_i."""
    rows, d_q = c_q.shape
    zeros = lambda n: torch.zeros((n, d_q), dtype=c_q.dtype)
    _, qn, _ = oracle.project(c_q.cpu().reshape(rows, 1, d_q), zeros(8), zeros(d_r), w_q.cpu(), H,
                              d_h, 0)
    return oracle.absorb_q(qn, w_uk.cpu())


def test_fp32_merged_query_tiny_widths():
    rows, H, d_h, d_r, d_c, d_q = 5, 8, 32, 16, 64, 96
    g = torch.Generator().manual_seed(75)
    w_uk = torch.randn((H, d_h, d_c), generator=g) / 8
    w_q = torch.randn((H * (d_h + d_r), d_q), generator=g) / 10
    c_q = torch.randn((rows, d_q), generator=g)
    w_m = mla.fold_q_weights(w_uk.cuda(), w_q.cuda(), d_r)
    q_lat = mla.absorb_q_merged(c_q.cuda(), w_m)
    torch.cuda.synchronize()
    ref = _unmerged_q_lat(c_q, w_q, w_uk, H, d_h, d_r)
    assert np.abs(q_lat.cpu().double().numpy() - ref).max() <= FP32_MAX


def test_bf16_merged_query_model_widths():
    """64 query rows, 16 heads of d_h 128 / d_c 512, compressed query 1536
    wide: the merged weight [1536, 16, 512] against W^UQ and W^UK apart."""
    rows, H, d_h, d_r, d_c, d_q = 64, 16, 128, 64, 512, 1536
    g = torch.Generator().manual_seed(76)
    w_uk = workloads.weight((H, d_h, d_c), d_c, g, "cpu", torch.bfloat16)
    w_q = workloads.weight((H * (d_h + d_r), d_q), d_q, g, "cpu", torch.bfloat16)
    c_q = torch.randn((rows, d_q), generator=g).to(torch.bfloat16)
    w_m = mla.fold_q_weights(w_uk.cuda(), w_q.cuda(), d_r)
    q_lat = mla.absorb_q_merged(c_q.cuda(), w_m)
    torch.cuda.synchronize()
    ref = _unmerged_q_lat(c_q, w_q, w_uk, H, d_h, d_r).reshape(rows, H, d_c)
    got = q_lat.float().cpu().double().numpy()
    err, excess, _, _ = o_excess(got, ref)
    fro = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    print(f"[parity] merged query: max|q-q*| {err:.3e}, rel fro {fro:.3e}")
    assert excess <= 0 and fro <= O_FRO
    # sampled entries of the fold against the fp64 product of the bf16 weights
    gs = torch.Generator().manual_seed(77)
    k = torch.randint(0, d_q, (64,), generator=gs).tolist()
    i = torch.randint(0, H, (64,), generator=gs).tolist()
    c = torch.randint(0, d_c, (64,), generator=gs).tolist()
    wm = w_m.cpu().double()
    for kk, ii, cc in zip(k, i, c):
        exact = float((w_uk[ii, :, cc].double() * w_q[ii * (d_h + d_r):ii * (d_h + d_r) + d_h, kk].double()).sum())
        assert abs(float(wm[kk, ii, cc]) - exact) <= REL * abs(exact) + 1e-6
