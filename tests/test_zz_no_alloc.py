"""mla_decode_attn_noalloc against mla_decode_attn (needs a B300).

The no-allocation entry point serves callers that cannot allocate device
memory (a host that owns all GPU memory and passes in only inputs and
outputs, or a path where an allocation could block the device); its
scratch is a fixed array inside the library.  It must give the same o and
lse as the regular entry point with a caller-owned workspace, call after
call, although every call reuses that one array.  This file sorts last so
that a run stopping at the first failure has run every other test first;
it also passes on its own in a fresh process.
"""

from __future__ import annotations

import pytest
import torch

from mla_latent_kv_71_b300 import mla, workloads

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.library()
    mla.get_device_status()
    yield
    assert mla.get_device_status()[0] == 0


def _same(case):
    """Both entry points on one case: the same kernels with the same plan, so
    the results must agree bit for bit (a stale value left in the shared
    scratch by an earlier call would show up here)."""
    o_ref, lse_ref = mla.decode_attn(case.q_lat, case.q_pe, case.pool, case.page_table,
                                     case.seq_lens, case.scale, causal=case.causal)
    o, lse = mla.decode_attn_noalloc(case.q_lat, case.q_pe, case.pool, case.page_table,
                                     case.seq_lens, case.scale, causal=case.causal)
    torch.cuda.synchronize()
    assert mla.get_device_status()[0] == 0
    assert torch.equal(o, o_ref), f"o differs in {(o != o_ref).sum().item()} elements"
    assert torch.equal(lse, lse_ref)


def test_noalloc_matches_decode_attn_on_two_calls_in_a_row():
    assert mla.noalloc_max_bytes() > 0
    # two different batches, so the second call must not depend on what the
    # first one left in the shared scratch; both cut sequences across SMs
    cases = [
        workloads.decode_case(24, 1, 128, 512, 64,
                              [int(x) for x in torch.randint(1, 3000, (24,),
                                                             generator=torch.Generator().manual_seed(5))],
                              seed=61, device="cuda"),
        workloads.decode_case(6, 2, 128, 512, 64, [700, 65, 1, 2048, 130, 999], seed=62,
                              device="cuda", hot_frac=0.01),
    ]
    for case in cases:
        B, T, H, d_c = case.q_lat.shape
        assert mla.decode_workspace_size(B, T, H, d_c) <= mla.noalloc_max_bytes()
        _same(case)


def test_noalloc_at_the_largest_batch_its_scratch_holds():
    """The largest batch whose scratch fits, with short ragged sequences cut
    between SMs up to the last unit: partial results land at the far end of
    the fixed array."""
    limit = mla.noalloc_max_bytes()
    B = 1
    while mla.decode_workspace_size(B + 1, 1, 128, 512) <= limit:
        B += 1
    assert mla.decode_workspace_size(B, 1, 128, 512) > limit - (1 << 20)  # within a slot
    lens = [int(x) for x in torch.randint(1, 400, (B,), generator=torch.Generator().manual_seed(64))]
    case = workloads.decode_case(B, 1, 128, 512, 64, lens, seed=65, device="cuda")
    plan = mla.decode_plan(lens, 1, 128, case.page_table.shape[1])
    assert max(p["slot"] for p in plan) >= B  # a slot in the last stretch of the array
    _same(case)
    _same(case)  # and again over what the first call left behind


def test_noalloc_rejects_a_shape_beyond_its_scratch():
    # enough (sequence, token) units that the partial-result scratch exceeds
    # the fixed array: refused on the host, nothing launched
    B, T = 4, 64
    assert mla.decode_workspace_size(B, T, 128, 512) > mla.noalloc_max_bytes()
    case = workloads.decode_case(B, T, 128, 512, 64, [T] * B, seed=63, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        mla.decode_attn_noalloc(case.q_lat, case.q_pe, case.pool, case.page_table, case.seq_lens,
                                case.scale, causal=True)
    assert e.value.code == 2  # MLA_ERR_UNSUPPORTED
