"""Token-range sharding of long sequences over several GPUs.

Under tensor parallelism the latent cache cannot be split by head, because
every head reads all of it: it has to be copied to every GPU or exchanged
([llms] "Hardware Trade-offs and Tensor Parallelism").  Splitting by token
range instead keeps one copy: rank r of W holds a contiguous range of each
sequence's pages, attends over them alone, and the ranks exchange one pair
(o_r, lse_r) per (sequence, query token, head) -- the normalised result
over its range and that range's log-sum-exp.  The log-sum-exp merge

    lse = ln sum_r e^{lse_r},    o = sum_r e^{lse_r - lse} o_r

is exact, so the merged result equals attention over the whole sequence up
to rounding.  Per rank and step the exchange is B*T*H*(d_c + 1) fp32 values
(256.5 KB per sequence at H = 128, d_c = 512), against the cache bytes the
rank reads.

Shard boundaries are page-aligned and as even as the page count allows.
With T causal query tokens (query t at position len - T + t), every shard
but the one holding the sequence's end must lie wholly before the first
query position, so that each of those shards is visible in full to every
query; the boundaries are pulled down to make it so.  Then ranks 0..W-2
attend without masking and rank W-1 (which always holds the end) with the
causal rule of the decode call.

This module is host logic: the per-rank attention and the merge are the
library's calls (mla_decode_attn_partial, mla_combine_splits) and the
exchange is one torch.distributed all-gather (NCCL between GPUs).
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

PAGE = 64


@dataclass
class Shard:
    """One rank's part of a batch: its pages of every sequence."""
    page_table: torch.Tensor   # [B, max_local_pages] int32, -1 past each sequence's last page
    seq_lens: torch.Tensor     # [B] int32 positions of each sequence held by this rank
    causal: bool               # whether this rank applies the causal rule (rank W-1 only)
    first_page: list           # [B] index of the rank's first page within each sequence


def page_bounds(length: int, T: int, world: int, page: int = PAGE) -> list[int]:
    """Page boundaries e_0 = 0 <= e_1 <= ... <= e_W = pages of one sequence:
    rank r holds pages [e_r, e_{r+1}).  Inner boundaries lie at or before the
    page holding the first query position (len - T), so that only the last
    rank's pages can hold positions some query must not see."""
    n = -(-length // page) if length > 0 else 0
    cap = max(length - T + 1, 0) // page  # pages wholly before position len - T + 1
    return [0] + [min(r * n // world, cap) for r in range(1, world)] + [n]


def shard_batch(seq_lens, page_table: torch.Tensor, T: int, world: int, rank: int,
                page: int = PAGE) -> Shard:
    """Rank `rank`'s shard of a batch given by host lengths and a page table."""
    lens = [int(x) for x in seq_lens]
    B = len(lens)
    table = page_table.cpu()
    rows, counts, first = [], [], []
    for b, L in enumerate(lens):
        e = page_bounds(L, T, world, page)
        p0, p1 = e[rank], e[rank + 1]
        rows.append(table[b, p0:p1])
        first.append(p0)
        if rank < world - 1:
            counts.append((p1 - p0) * page)  # whole pages, all before the queries
        else:
            counts.append(max(L - p0 * page, 0) if p1 > p0 else 0)
    width = max(1, max(r.numel() for r in rows))
    local = torch.full((B, width), -1, dtype=torch.int32)
    for b, r in enumerate(rows):
        local[b, :r.numel()] = r
    return Shard(page_table=local.to(page_table.device),
                 seq_lens=torch.tensor(counts, dtype=torch.int32, device=page_table.device),
                 causal=(rank == world - 1) and T > 1, first_page=first)


def _all_gather(x: torch.Tensor, world: int, group=None) -> torch.Tensor:
    """[world, *x.shape]: every rank's x, in rank order (the one exchange)."""
    import torch.distributed as dist
    parts = [torch.empty_like(x) for _ in range(world)]
    dist.all_gather(parts, x.contiguous(), group=group)
    return torch.stack(parts)


def sharded_decode(q_lat, q_pe, kv_pool, shard: Shard, scale: float, world: int, group=None,
                   partial_fn=None, combine_fn=None, gather_fn=None):
    """Attention over a batch whose sequences are sharded by token range.

    Every rank calls this with the same queries and its own Shard (and the
    pool holding its pages).  Returns (o, lse) of the whole sequences, the
    same on every rank: o [B, T, H, d_c] in the query's type, lse [B, T, H].
    partial_fn / combine_fn / gather_fn default to the library's
    decode_attn_partial and combine_splits and a torch.distributed
    all-gather; they are parameters only so that the exchange can be run
    against other implementations of the same two steps.
    """
    if partial_fn is None or combine_fn is None:
        from . import mla
        partial_fn = partial_fn or mla.decode_attn_partial
        combine_fn = combine_fn or mla.combine_splits
    gather_fn = gather_fn or (lambda x: _all_gather(x, world, group))
    B, T, H, d_c = q_lat.shape
    o_r, lse_r = partial_fn(q_lat, q_pe, kv_pool, shard.page_table, shard.seq_lens, scale,
                            causal=shard.causal)
    o_all = gather_fn(o_r.reshape(B * T * H, d_c))      # [W, rows, d_c] fp32
    lse_all = gather_fn(lse_r.reshape(B * T * H))        # [W, rows]
    o, lse = combine_fn(o_all, lse_all, out_dtype=q_lat.dtype)
    return o.reshape(B, T, H, d_c), lse.reshape(B, T, H)
