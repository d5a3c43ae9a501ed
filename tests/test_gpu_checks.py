"""The debug build (needs a B300): libmla_checks.so, built with MLA_CHECKS=1.

Its kernels check their own work split against the shapes (the decode's
page pieces and partial slots, the merge's piece ranges, the GEMM's items,
the prefill's key blocks) and raise the device status word on a violation;
they also fill their shared memory with NaN (all-ones bytes) before use, so
that a read of a byte no copy wrote shows up in the results.  Each case
runs in a child process with MLA_CHECKS=1 (the binding then loads the debug
library), compares every output element with the fp64 oracle at the usual
bars, and requires a clean device status.  Outputs are NaN-filled before
each call as well, so an element the kernels never write fails the check.
"""

from __future__ import annotations

import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
import numpy as np
import torch
sys.path.insert(0, ROOT)
import oracle
from mla_latent_kv_71_b300 import mla, workloads
from tests.bars import LSE_MAX, O_FRO, o_excess

assert mla.CHECKS and mla.LIB_PATH.endswith("libmla_checks.so")
dev = torch.device("cuda", 0)


def nan_like(t):
    return torch.full_like(t, float("nan"))


def check(got, ref, what, lse=None, lse_ref=None):
    got = got.float().cpu().numpy().reshape(ref.shape)
    assert np.isfinite(got).all(), what + ": an output element was not written"
    err, excess, _, _ = o_excess(got, ref)
    assert excess <= 0, f"{what}: max err {err:.3e}"
    assert np.linalg.norm(got - ref) <= O_FRO * np.linalg.norm(ref), what
    if lse is not None:
        l = lse.cpu().numpy().reshape(lse_ref.shape)
        fin = np.isfinite(lse_ref)
        assert (np.isneginf(l) == ~fin).all(), what
        assert np.abs(l[fin] - lse_ref[fin]).max() <= LSE_MAX, what
    code, detail = mla.get_device_status()
    assert code == 0, f"{what}: device status {code} detail {detail:#x}"
    print("ok", what, f"{err:.2e}")


def decode(lens, T, H, host, what):
    case = workloads.decode_case(len(lens), T, H, 512, 64, lens, seed=91, device=dev)
    o, lse = nan_like(case.q_lat), torch.full(case.q_lat.shape[:3], float("nan"), device=dev)
    mla.decode_attn(case.q_lat, case.q_pe, case.pool, case.page_table, case.seq_lens, case.scale,
                    causal=T > 1, o=o, lse=lse, seq_lens_host=case.seq_lens.cpu() if host else None)
    torch.cuda.synchronize()
    c = workloads.DecodeCase(*(t.cpu() for t in (case.q_lat, case.q_pe, case.pool, case.page_table,
                                                 case.seq_lens)), case.scale, T > 1)
    o_ref, lse_ref = oracle.decode_attn(c.q_lat, c.q_pe, c.pool, c.page_table, c.seq_lens, c.scale,
                                        causal=c.causal)
    check(o, o_ref, what, lse, lse_ref)


# cut units merged across clusters, with an empty sequence
decode([int(x) for x in torch.randint(1, 3000, (24,), generator=torch.Generator().manual_seed(3))] + [0],
       1, 128, False, "decode cut and merged")
# one cluster per sequence (equal lengths, host lengths)
decode([700] * 20, 1, 128, True, "decode one cluster per sequence")
# two causal tokens, two head groups
decode([300, 65, 129], 2, 200, True, "decode two tokens, 200 heads")

# the GEMM: query absorption and the split-K output projection
g = torch.Generator(device=dev).manual_seed(92)
qn = (torch.randn((48, 16, 128), generator=g, device=dev)).to(torch.bfloat16)
w_uk, w_uv, w_o = workloads.projection_weights(16, 128, 512, 1024, seed=93, device=dev)
q_lat = torch.full((48, 16, 512), float("nan"), device=dev).to(torch.bfloat16)
mla.absorb_q(qn, w_uk, q_lat)
torch.cuda.synchronize()
check(q_lat, oracle.absorb_q(qn.cpu(), w_uk.cpu()), "absorb_q")
o = (torch.randn((48, 16, 512), generator=g, device=dev) * 0.05).to(torch.bfloat16)
out = mla.out_proj(o, w_uv, w_o)
torch.cuda.synchronize()
ref, _ = oracle.out_proj(o.cpu(), w_uv.cpu(), w_o.cpu())
check(out, ref, "out_proj")

# the query projection written by the GEMM's epilogue (heads split, q^R rotated)
N, H, d_h, d_r, d_q = 40, 128, 128, 64, 1536
ch = torch.randn((N, d_q), generator=g, device=dev).to(torch.bfloat16)
w_q = workloads.weight((H * (d_h + d_r), d_q), d_q, g, dev, torch.bfloat16)
pos = torch.randint(0, 100001, (N,), generator=g, device=dev, dtype=torch.int32)
qn = torch.full((N, H, d_h), float("nan"), device=dev).to(torch.bfloat16)
qp = torch.full((N, H, d_r), float("nan"), device=dev).to(torch.bfloat16)
mla.project_q(ch, w_q, pos, H, d_h, d_r, qn, qp)
torch.cuda.synchronize()
_, qn_ref, qp_ref = oracle.project(ch.cpu().reshape(N, 1, d_q), torch.zeros((2, d_q), dtype=torch.bfloat16),
                                   torch.zeros((d_r, d_q), dtype=torch.bfloat16), w_q.cpu(), H, d_h, qpos=0)
for n, ps in enumerate(pos.tolist()):
    for i in range(H):
        qp_ref[n, i] = oracle.rope(qp_ref[n, i], ps)
check(qn, qn_ref, "project_q content")
check(qp, qp_ref, "project_q rotated")

# the prefill attention (causal, a ragged last block)
case = workloads.prefill_case(1, 300, 4, d=1024, seed=94, device=dev)
k, v = mla.prefill_expand(case.kv, case.w_uk, case.w_uv)
u, lse = mla.prefill_attn(case.q_nope, case.q_pe, k, case.kv, v, case.L, case.scale, True)
torch.cuda.synchronize()
u_ref, lse_ref = oracle.prefill_attn(case.q_nope.cpu(), case.q_pe.cpu(), k.cpu(), case.kv.cpu(), v.cpu(),
                                     case.L, case.scale, causal=True, k_pe_off=512)
check(u, u_ref.reshape(-1, 128), "prefill attention", lse, lse_ref.reshape(-1))
print("all ok")
'''


def test_debug_build_checks_and_parity():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = os.path.join(ROOT, "mla_latent_kv_71_b300", "libmla_checks.so")
    if not os.path.exists(lib):
        from mla_latent_kv_71_b300 import build
        build.build(checks=True)
    env = dict(os.environ, MLA_CHECKS="1")
    r = subprocess.run([sys.executable, "-c", f"ROOT = {ROOT!r}\n" + CHILD], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    print(r.stdout[-4000:])
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "all ok" in r.stdout
