"""Seeded synthetic inputs for MLA absorbed decode.

This module only draws random numbers and lays them out (rounding to the
storage type, building page tables); it holds none of the method's
arithmetic.  Both the CUDA path's tests and the oracle's tests take their
inputs from here, so the two sides see identical bit patterns.

Recipe (all values are drawn in fp32 from a ``torch.Generator`` seeded as
stated, then rounded to the storage type with round-to-nearest-even):

* Decode batches: q_lat, q_pe, then the pool rows [c ; k_pe] are drawn
  N(0, 1) in that order.  Each sequence owns ceil(len/page) pages; the pool
  holds exactly those pages, placed at a random permutation drawn from a
  second generator seeded with ``seed + 1000``.  Page-table entries past a
  sequence's last page are -1.  Optionally a fraction of each sequence's
  rows has its latent part (the first d_c values) scaled by a power of two.
* Ragged lengths are drawn uniformly from [1, max_len] with the stated seed.
* Projection weights are drawn N(0, 1/fan_in), fan_in being the input width
  of the map; hidden states are N(0, 1).
* Prefill batches (every token a query): cache rows [c ; k^R], then q^C and
  q^R, drawn N(0, 1) in that order, then W^UK, W^UV, W^O as above.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

PAGE = 64


@dataclass
class DecodeCase:
    """One decode step's inputs (tensors on ``device``)."""
    q_lat: torch.Tensor          # [B, T, H, d_c]
    q_pe: torch.Tensor           # [B, T, H, d_r]
    pool: torch.Tensor           # [P, page, d_c + d_r]
    page_table: torch.Tensor     # [B, max_pages] int32, -1 past the end
    seq_lens: torch.Tensor       # [B] int32
    scale: float
    causal: bool
    extra: dict = field(default_factory=dict)

    @property
    def dims(self):
        B, T, H, d_c = self.q_lat.shape
        return dict(B=B, T=T, H=H, d_c=d_c, d_r=self.q_pe.shape[3], page=self.pool.shape[1],
                    max_pages=self.page_table.shape[1], num_pages=self.pool.shape[0])


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def ragged_lengths(B: int, max_len: int, seed: int) -> list[int]:
    """B lengths drawn uniformly from [1, max_len] (inclusive)."""
    g = _gen(seed, "cpu")
    return torch.randint(1, max_len + 1, (B,), generator=g).tolist()


def decode_case(B: int, T: int, H: int, d_c: int, d_r: int, lens, *, page: int = PAGE,
                seed: int = 0, dtype=torch.bfloat16, device="cpu", scale: float | None = None,
                d_h: int = 128, causal: bool | None = None, hot_frac: float = 0.0,
                hot_factor: float = 8.0) -> DecodeCase:
    """Random decode batch with a paged latent cache.

    lens: per-sequence cache lengths (list of B ints).  scale defaults to
    1/sqrt(d_h + d_r).  causal defaults to T > 1.  hot_frac > 0 scales the
    latent part of round(hot_frac * len) distinct rows per sequence by
    hot_factor (exact in binary floating point for powers of two).
    """
    lens = [int(x) for x in lens]
    assert len(lens) == B
    g = _gen(seed, device)
    q_lat = torch.randn((B, T, H, d_c), generator=g, device=device, dtype=torch.float32)
    q_pe = torch.randn((B, T, H, d_r), generator=g, device=device, dtype=torch.float32)
    n_pages = [max(0, math.ceil(n / page)) for n in lens]
    P = sum(n_pages)
    max_pages = max(1, max(n_pages) if n_pages else 1)
    pool = torch.randn((max(P, 1), page, d_c + d_r), generator=g, device=device,
                       dtype=torch.float32)
    gp = _gen(seed + 1000, "cpu")
    perm = torch.randperm(max(P, 1), generator=gp)
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    off = 0
    for b in range(B):
        table[b, :n_pages[b]] = perm[off:off + n_pages[b]].to(torch.int32)
        off += n_pages[b]
    if hot_frac > 0.0:
        gh = _gen(seed + 2000, "cpu")
        flat = pool.view(-1, d_c + d_r)
        for b in range(B):
            k = int(round(hot_frac * lens[b]))
            if k == 0:
                continue
            rows = torch.randperm(lens[b], generator=gh)[:k]
            phys = table[b, rows // page].to(torch.int64) * page + rows % page
            flat[phys.to(device), :d_c] *= hot_factor
    if scale is None:
        scale = 1.0 / math.sqrt(d_h + d_r)
    return DecodeCase(
        q_lat=q_lat.to(dtype), q_pe=q_pe.to(dtype), pool=pool.to(dtype),
        page_table=table.to(device), seq_lens=torch.tensor(lens, dtype=torch.int32,
                                                           device=device),
        scale=float(scale), causal=(T > 1) if causal is None else bool(causal))


def weight(shape, fan_in: int, g: torch.Generator, device, dtype) -> torch.Tensor:
    w = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return (w * (1.0 / math.sqrt(fan_in))).to(dtype)


def projection_weights(H: int, d_h: int, d_c: int, d: int, *, seed: int, device="cpu",
                       dtype=torch.bfloat16):
    """W^UK, W^UV [H, d_h, d_c] (fan_in d_c) and W^O [d, H*d_h] (fan_in H*d_h)."""
    g = _gen(seed, device)
    w_uk = weight((H, d_h, d_c), d_c, g, device, dtype)
    w_uv = weight((H, d_h, d_c), d_c, g, device, dtype)
    w_o = weight((d, H * d_h), H * d_h, g, device, dtype)
    return w_uk, w_uv, w_o


def q_nope(B: int, T: int, H: int, d_h: int, *, seed: int, device="cpu",
           dtype=torch.bfloat16) -> torch.Tensor:
    g = _gen(seed, device)
    return torch.randn((B, T, H, d_h), generator=g, device=device,
                       dtype=torch.float32).to(dtype)


@dataclass
class PrefillCase:
    """B sequences of L tokens, every token a query (tensors on ``device``)."""
    kv: torch.Tensor       # [B*L, d_c + d_r] cache rows [c ; k^R]
    q_nope: torch.Tensor   # [B*L, H, d_h]
    q_pe: torch.Tensor     # [B*L, H, d_r]
    w_uk: torch.Tensor     # [H, d_h, d_c]
    w_uv: torch.Tensor     # [H, d_h, d_c]
    w_o: torch.Tensor      # [d, H*d_h]
    B: int
    L: int
    scale: float


def prefill_case(B: int, L: int, H: int, *, d_h: int = 128, d_c: int = 512, d_r: int = 64,
                 d: int = 7168, seed: int = 0, device="cpu", dtype=torch.bfloat16) -> PrefillCase:
    g = _gen(seed, device)
    kv = torch.randn((B * L, d_c + d_r), generator=g, device=device, dtype=torch.float32)
    qn = torch.randn((B * L, H, d_h), generator=g, device=device, dtype=torch.float32)
    qp = torch.randn((B * L, H, d_r), generator=g, device=device, dtype=torch.float32)
    w_uk = weight((H, d_h, d_c), d_c, g, device, dtype)
    w_uv = weight((H, d_h, d_c), d_c, g, device, dtype)
    w_o = weight((d, H * d_h), H * d_h, g, device, dtype)
    return PrefillCase(kv.to(dtype), qn.to(dtype), qp.to(dtype), w_uk, w_uv, w_o, B, L,
                       1.0 / math.sqrt(d_h + d_r))


def tiny_model(seed: int = 0, device="cpu"):
    """The tiny fp32 model: B=2, d=256, H=8, d_h=32, d_c=64, d_r=16, L=128.

    Returns a dict of hidden states h [B, L, d] ~ N(0, 1) and the weights
    W^DKV [d_c, d], W^KR [d_r, d], W^Q [H*(d_h+d_r), d], W^UK, W^UV
    [H, d_h, d_c] and W^O [d, H*d_h], each N(0, 1/fan_in), all fp32.
    """
    B, d, H, d_h, d_c, d_r, L = 2, 256, 8, 32, 64, 16, 128
    g = _gen(seed, device)
    f32 = torch.float32
    h = torch.randn((B, L, d), generator=g, device=device, dtype=f32)
    w_dkv = weight((d_c, d), d, g, device, f32)
    w_kr = weight((d_r, d), d, g, device, f32)
    w_q = weight((H * (d_h + d_r), d), d, g, device, f32)
    w_uk = weight((H, d_h, d_c), d_c, g, device, f32)
    w_uv = weight((H, d_h, d_c), d_c, g, device, f32)
    w_o = weight((d, H * d_h), H * d_h, g, device, f32)
    return dict(B=B, d=d, H=H, d_h=d_h, d_c=d_c, d_r=d_r, L=L, h=h, w_dkv=w_dkv, w_kr=w_kr,
                w_q=w_q, w_uk=w_uk, w_uv=w_uv, w_o=w_o, rope_base=10000.0,
                scale=1.0 / math.sqrt(d_h + d_r))


# ----------------------------------------------------------- named workloads
#
# The decode workloads the library is measured and checked on.  Shapes follow
# DeepSeek-V2/V3 attention (H=128 heads, d_h=128, d_c=512, d_r=64) unless stated.

WORKLOADS = {
    # tiny fp32 model; decode inputs at its sizes for the fp32 kernels
    "tiny_fp32": dict(B=2, T=1, H=8, d_h=32, d_c=64, d_r=16, lens=[128, 128], seed=0,
                      dtype="fp32"),
    # uniform decode batch: the headline workload
    "decode_b64_h128_l4096": dict(B=64, T=1, H=128, d_h=128, d_c=512, d_r=64,
                                  lens=[4096] * 64, seed=0, dtype="bf16"),
    # ragged serving batch, lengths U[1, 16384] with seed 1
    "ragged_b128_l16k": dict(B=128, T=1, H=128, d_h=128, d_c=512, d_r=64,
                             lens=("ragged", 16384, 1), seed=1, dtype="bf16"),
    # long context, 1% of latent rows scaled by 8
    "long_b4_l128k": dict(B=4, T=1, H=128, d_h=128, d_c=512, d_r=64, lens=[131072] * 4,
                          seed=0, dtype="bf16", hot_frac=0.01),
    # two causal query tokens per sequence, end to end with projections (d=7168)
    "mtp_b32_t2_l8192": dict(B=32, T=2, H=128, d_h=128, d_c=512, d_r=64, lens=[8192] * 32,
                             seed=0, dtype="bf16", d=7168, e2e=True),
    # 16 heads, long cache, end to end with projections (d=7168)
    "smallhead_b64_h16_l32k": dict(B=64, T=1, H=16, d_h=128, d_c=512, d_r=64,
                                   lens=[32768] * 64, seed=0, dtype="bf16", d=7168, e2e=True),
}


def workload_lens(spec) -> list[int]:
    lens = spec["lens"]
    if isinstance(lens, tuple) and lens[0] == "ragged":
        return ragged_lengths(spec["B"], lens[1], lens[2])
    return list(lens)


def make_workload(name: str, device="cpu", B: int | None = None) -> DecodeCase:
    """Decode inputs of a named workload (optionally only its first B sequences)."""
    spec = WORKLOADS[name]
    lens = workload_lens(spec)
    if B is not None:
        lens = lens[:B]
    nb = len(lens)
    dtype = torch.float32 if spec["dtype"] == "fp32" else torch.bfloat16
    case = decode_case(nb, spec["T"], spec["H"], spec["d_c"], spec["d_r"], lens,
                       seed=spec["seed"], dtype=dtype, device=device, d_h=spec["d_h"],
                       hot_frac=spec.get("hot_frac", 0.0))
    if spec.get("e2e"):
        case.extra["q_nope"] = q_nope(nb, spec["T"], spec["H"], spec["d_h"],
                                      seed=spec["seed"] + 3000, device=device, dtype=dtype)
        w_uk, w_uv, w_o = projection_weights(spec["H"], spec["d_h"], spec["d_c"], spec["d"],
                                             seed=spec["seed"] + 4000, device=device,
                                             dtype=dtype)
        case.extra.update(w_uk=w_uk, w_uv=w_uv, w_o=w_o)
    return case
