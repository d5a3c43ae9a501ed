"""Token-range sharding on the GPU (needs a B300).

mla_decode_attn_partial against the oracle, and the sharded decode of
mla_latent_kv_71_b300.shard with W ranks emulated one after another on the
one GPU: each "rank" runs the partial call on its page range of every
sequence, the partials are stacked in rank order (what the all-gather
returns on every rank) and mla_combine_splits merges them.  No rank waits
on another, so running them in turn on one device is the same computation.
The merged result must meet the decode bars against the oracle's attention
over the whole sequences.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_71_b300 import mla, shard, workloads
from tests.bars import LSE_MAX, O_FRO, o_excess

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.library()
    yield


def _oracle(case, table=None, lens=None, causal=None):
    t = case.page_table if table is None else table
    n = case.seq_lens if lens is None else lens
    c = case.causal if causal is None else causal
    return oracle.decode_attn(case.q_lat.cpu(), case.q_pe.cpu(), case.pool.cpu(), t.cpu(),
                              n.cpu(), case.scale, causal=c)


def _check(o, lse, o_ref, lse_ref, what, case):
    got = o.float().cpu().numpy().reshape(o_ref.shape)
    c = workloads.DecodeCase(case.q_lat.cpu(), case.q_pe.cpu(), case.pool.cpu(),
                             case.page_table.cpu(), case.seq_lens.cpu(), case.scale, case.causal)
    spread = lambda rows: oracle.weight_spread(c.q_lat, c.q_pe, c.pool, c.page_table, c.seq_lens,
                                               c.scale, causal=c.causal, sel=rows)
    err, excess, _, _ = o_excess(got, o_ref, spread)
    fro = np.linalg.norm(got - o_ref) / np.linalg.norm(o_ref)
    lse = lse.cpu().numpy().reshape(lse_ref.shape)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin), what
    lerr = np.abs(lse[fin] - lse_ref[fin]).max()
    print(f"[parity] {what}: max|o-o*| {err:.3e}, rel fro {fro:.3e}, max|lse-lse*| {lerr:.3e}")
    assert excess <= 0 and fro <= O_FRO and lerr <= LSE_MAX, what


def test_partial_decode_writes_fp32_o():
    case = workloads.decode_case(3, 1, 128, 512, 64, [1000, 1, 4100], seed=92, device="cuda",
                                 hot_frac=0.01)
    o, lse = mla.decode_attn_partial(case.q_lat, case.q_pe, case.pool, case.page_table,
                                     case.seq_lens, case.scale)
    torch.cuda.synchronize()
    assert o.dtype == torch.float32 and mla.get_device_status()[0] == 0
    o_ref, lse_ref = _oracle(case)
    _check(o, lse, o_ref, lse_ref, "partial fp32 o", case)
    # rounding the fp32 result to bf16 (to nearest even) gives the bf16
    # call's result: both round the same fp32 value O / l (or the same
    # merge of partials) once
    o_bf, lse_bf = mla.decode_attn(case.q_lat, case.q_pe, case.pool, case.page_table,
                                   case.seq_lens, case.scale)
    torch.cuda.synchronize()
    assert torch.equal(lse, lse_bf)
    assert torch.equal(o.to(torch.bfloat16), o_bf)


@pytest.mark.parametrize("T,world", [(1, 2), (1, 4), (2, 3)])
def test_sharded_decode_emulated_ranks(T, world):
    lens = [20000, 5000, 70, 1]
    case = workloads.decode_case(len(lens), T, 128, 512, 64, lens, seed=93 + world, device="cuda")
    parts = []
    for r in range(world):
        sh = shard.shard_batch(lens, case.page_table, T, world, r)
        parts.append(mla.decode_attn_partial(case.q_lat, case.q_pe, case.pool, sh.page_table,
                                             sh.seq_lens, case.scale, causal=sh.causal))
    # the one exchange step, as every rank would see it after the all-gather
    gathered = iter([torch.stack([p[0].reshape(-1, 512) for p in parts]),
                     torch.stack([p[1].reshape(-1) for p in parts])])
    sh0 = shard.shard_batch(lens, case.page_table, T, world, 0)
    o, lse = shard.sharded_decode(case.q_lat, case.q_pe, case.pool, sh0, case.scale, world,
                                  gather_fn=lambda x: next(gathered))
    torch.cuda.synchronize()
    assert mla.get_device_status()[0] == 0
    o_ref, lse_ref = _oracle(case)
    _check(o, lse, o_ref, lse_ref, f"sharded T={T} W={world}", case)
