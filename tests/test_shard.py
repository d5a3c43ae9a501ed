"""Token-range sharding of long sequences (mla_latent_kv_71_b300.shard) on
CPU ranks: two gloo processes each attend over their page range of every
sequence, all-gather their (o, lse) partials -- the one exchange step -- and
merge them by log-sum-exp.  The per-rank attention and the merge are the
fp64 oracle's here (the ranks have no GPU); the result must equal the
oracle's attention over the whole sequences.  The boundary rule is checked
directly on the host."""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from mla_latent_kv_71_b300 import shard

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("length,T,world", [(1000, 1, 2), (129, 2, 2), (65, 2, 3), (64, 3, 4),
                                            (1, 1, 2), (0, 1, 2), (8193, 2, 4)])
def test_page_bounds_cover_every_page_once_and_keep_the_queries_last(length, T, world):
    e = shard.page_bounds(length, T, world)
    n = -(-length // 64)
    assert e[0] == 0 and e[-1] == n and all(a <= b for a, b in zip(e, e[1:]))
    # every inner boundary lies at or before the first query position
    assert all(64 * x <= max(length - T + 1, 0) for x in e[1:-1])
    if n:
        assert e[-2] < e[-1]  # the last rank holds the sequence's end


def _oracle_partial(q_lat, q_pe, pool, table, lens, scale, causal=False):
    import oracle
    o, lse = oracle.decode_attn(q_lat, q_pe, pool, table, lens, scale, causal=causal)
    return torch.from_numpy(o).reshape(q_lat.shape), torch.from_numpy(lse).reshape(q_lat.shape[:3])


def _oracle_combine(o_all, lse_all, out_dtype=None):
    import oracle
    o, lse = oracle.combine(o_all.numpy(), lse_all.numpy())
    return torch.from_numpy(o), torch.from_numpy(lse)


def _case():
    from mla_latent_kv_71_b300 import workloads
    # two causal query tokens; lengths that leave ragged last pages, a
    # sequence shorter than one page per rank and one of a single token
    return workloads.decode_case(4, 2, 8, 64, 16, [700, 130, 70, 2], seed=91, d_h=32,
                                 dtype=torch.float32)


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    case = _case()
    sh = shard.shard_batch(case.seq_lens.tolist(), case.page_table, 2, world, rank)
    o, lse = shard.sharded_decode(case.q_lat, case.q_pe, case.pool, sh, case.scale, world,
                                  partial_fn=_oracle_partial, combine_fn=_oracle_combine)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, o.numpy(), lse.numpy(), sh.seq_lens.tolist()))


def test_sharded_decode_on_two_gloo_ranks_equals_whole_sequence_attention():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=240) for _ in range(world)), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0, p.exitcode
    case = _case()
    o_ref, lse_ref = _oracle_partial(case.q_lat, case.q_pe, case.pool, case.page_table,
                                     case.seq_lens, case.scale, causal=True)
    # the split really cut sequences: each rank held part of the longest one
    assert all(r[3][0] > 0 for r in res)
    for _, o, lse, _ in res:  # every rank ends with the whole-sequence result
        np.testing.assert_allclose(o, o_ref.numpy(), rtol=0, atol=1e-12)
        fin = np.isfinite(lse_ref.numpy())
        assert np.array_equal(np.isfinite(lse), fin)
        np.testing.assert_allclose(lse[fin], lse_ref.numpy()[fin], rtol=0, atol=1e-12)
