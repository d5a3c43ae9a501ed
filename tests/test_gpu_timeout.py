"""The bounded-wait failure path (needs a B300).

Every wait of a pipeline step in the library's kernels gives up after a
limit, raises MLA_ERR_TIMEOUT in the device status word and lets the kernel
wind down: the CTA waits for the copies and tensor-core products it issued
itself, frees its TMEM and exits.  These tests shorten the limit from the
host to 1 ns, so that a wait still open after the hardware's first
suspension gives up, and check that the call reports the timeout and that
the next call on the same context computes the right result.  Nothing is broken on purpose: no
arrival is skipped and no input is invalid; the waits simply give up early.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_71_b300 import mla, workloads
from tests.bars import LSE_MAX, O_FRO, o_excess

pytestmark = pytest.mark.gpu

MLA_ERR_TIMEOUT = 4


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.library()
    yield
    mla.set_wait_limit(0)


def _timed_out(fn, tries=3):
    """Run fn with a 1 ns wait limit until a call reports the timeout (at
    most `tries` calls); returns the last (status code, detail).  A wait
    only gives up when the hardware's first suspension inside try_wait ends
    before the phase completes, so a single call may see every wait met."""
    code, detail = 0, 0
    for _ in range(tries):
        mla.get_device_status()
        mla.set_wait_limit(1)
        try:
            fn()
            torch.cuda.synchronize()
            code, detail = mla.get_device_status()
        finally:
            mla.set_wait_limit(0)
        if code != 0:
            break
    return code, detail


def test_decode_wait_gives_up_and_the_next_call_is_correct():
    # 16 sequences of 4096: every cluster streams several pages, so some wait
    # is still open after its first try (a batch of a few pages can finish
    # every wait inside the first one, and then nothing gives up)
    case = workloads.decode_case(16, 1, 128, 512, 64, [4096] * 16, seed=81, device="cuda")
    args = (case.q_lat, case.q_pe, case.pool, case.page_table, case.seq_lens, case.scale)
    code, detail = _timed_out(lambda: mla.decode_attn(*args))
    assert code == MLA_ERR_TIMEOUT, (code, hex(detail))
    o, lse = mla.decode_attn(*args)
    torch.cuda.synchronize()
    assert mla.get_device_status()[0] == 0
    c = workloads.DecodeCase(*(t.cpu() for t in args[:5]), case.scale, False)
    o_ref, lse_ref = oracle.decode_attn(c.q_lat, c.q_pe, c.pool, c.page_table, c.seq_lens,
                                        c.scale)
    got = o.float().cpu().numpy().reshape(o_ref.shape)
    _, excess, _, _ = o_excess(got, o_ref)
    assert excess <= 0
    assert np.linalg.norm(got - o_ref) <= O_FRO * np.linalg.norm(o_ref)
    assert np.abs(lse.cpu().numpy().reshape(lse_ref.shape) - lse_ref).max() <= LSE_MAX


def test_split_k_projection_gives_up_and_its_counters_recover():
    """out_proj reduces W^O over split-K CTAs with arrival counters kept in
    the workspace; after a call whose waits gave up, the next calls with the
    same workspace must still reduce every tile exactly once."""
    rows, H, d = 16, 128, 7168
    g = torch.Generator(device="cuda").manual_seed(82)
    o = (torch.randn((rows, H, 512), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    _, w_uv, w_o = workloads.projection_weights(H, 128, 512, d, seed=83, device="cuda")
    need = mla.out_proj_workspace_size(rows, H, 128, d)
    assert need > 0  # split-K is in use
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    code, _ = _timed_out(lambda: mla.out_proj(o, w_uv, w_o, workspace=ws))
    assert code == MLA_ERR_TIMEOUT
    out1 = mla.out_proj(o, w_uv, w_o, workspace=ws)
    out2 = mla.out_proj(o, w_uv, w_o, workspace=ws)
    torch.cuda.synchronize()
    assert mla.get_device_status()[0] == 0
    assert torch.equal(out1, out2)
    ref, _ = oracle.out_proj(o.cpu(), w_uv.cpu(), w_o.cpu())
    got = out1.float().cpu().numpy()
    _, excess, _, _ = o_excess(got, ref)
    assert excess <= 0
    assert np.linalg.norm(got - ref) <= O_FRO * np.linalg.norm(ref)
