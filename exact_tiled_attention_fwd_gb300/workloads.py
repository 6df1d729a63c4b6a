"""Seeded synthetic inputs shaped like the pages' workloads.

Random numbers only: this module holds none of the attention arithmetic.  It
serves the tests (both the CUDA path and the float64 oracle read the very same
tensors) and bench.py.

Recipe (all values bf16 drawn i.i.d. from N(0, 1), then rounded to bf16):

  C1  dense   B=1,  H=1,  N=256,  d=64,  non-causal
  C2  dense   B=4,  H=16, N=2048, d=128, non-causal and causal
  C3  dense   B=1,  H=32, N=8192, d=128, non-causal and causal
  C4  varlen  16 sequences, lengths uniform integers in [128, 4096], H=32,
              d=64, causal inside each sequence
  C5  paged   B=64 single-token queries, H=32, d=128, KV lengths uniform
              integers in [512, 16384], 16-token pages, block_table a seeded
              random permutation of the pool's physical pages

Small tensors are drawn on the CPU with a seeded torch.Generator and copied
to the device, so any machine gets the same values; the C5 page pool (about
8.9 GB) is drawn directly on the device with a seeded CUDA generator.  Page
permutations and lengths always come from the CPU generator.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

PAGE_SIZE = 16


@dataclass(frozen=True)
class Dense:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    Hkv: int | None = None

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


CONFIGS = {
    "C1": Dense("C1", 1, 1, 256, 64, False),
    "C2": Dense("C2", 4, 16, 2048, 128, False),
    "C2c": Dense("C2c", 4, 16, 2048, 128, True),
    "C3": Dense("C3", 1, 32, 8192, 128, False),
    "C3c": Dense("C3c", 1, 32, 8192, 128, True),
}
VARLEN_C4 = dict(num_seqs=16, lo=128, hi=4096, H=32, d=64, causal=True)
PAGED_C5 = dict(B=64, H=32, d=128, lo=512, hi=16384, page_size=PAGE_SIZE)
# Prefix-cache continuation chunk: cached context plus a chunk of new tokens
# per sequence, attended through the page table (store_kvcache first).
CHUNK = dict(num_seqs=16, ctx_lo=512, ctx_hi=8192, new_lo=256, new_hi=2048, H=32, d=128, causal=True)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def randn_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    """i.i.d. N(0,1) rounded to bf16, drawn on the CPU, then moved."""
    t = torch.randn(shape, generator=_gen(seed), dtype=torch.float32).to(torch.bfloat16)
    return t.to(device)


def randn_bf16_device(shape, seed: int, device) -> torch.Tensor:
    """i.i.d. N(0,1) bf16 drawn directly on a CUDA device (large pools)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.bfloat16, device=device)


def sign_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    """i.i.d. uniform signs (+1 or -1) as bf16, drawn on the CPU, then moved.
    Used for key pools whose scores against a chosen key must be exact
    integers (the one-hot gather tests)."""
    t = torch.randint(0, 2, shape, generator=_gen(seed), dtype=torch.int16)
    return (t * 2 - 1).to(torch.bfloat16).to(device)


def sign_bf16_device(shape, seed: int, device) -> torch.Tensor:
    """i.i.d. uniform signs as bf16, drawn directly on a CUDA device."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randint(0, 2, shape, generator=g, dtype=torch.int16, device=device)
    return (t * 2 - 1).to(torch.bfloat16)


def dense_inputs(B, N, H, d, seed: int, device="cpu", Hkv=None):
    """q [B, N, H, d], k, v [B, N, Hkv, d] bf16."""
    Hkv = H if Hkv is None else Hkv
    q = randn_bf16((B, N, H, d), seed * 3 + 0, device)
    k = randn_bf16((B, N, Hkv, d), seed * 3 + 1, device)
    v = randn_bf16((B, N, Hkv, d), seed * 3 + 2, device)
    return q, k, v


def uniform_lengths(n: int, lo: int, hi: int, seed: int) -> list[int]:
    """n integers uniform in [lo, hi] (inclusive)."""
    return torch.randint(lo, hi + 1, (n,), generator=_gen(seed)).tolist()


def cu_seqlens(lengths) -> torch.Tensor:
    """int32 prefix sums [0, l0, l0+l1, ...] (the varlen boundary array)."""
    out = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    out[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return out


def varlen_inputs(lengths_q, H, d, seed: int, device="cpu", lengths_k=None, Hkv=None):
    """Packed q [total_q, H, d], k, v [total_k, Hkv, d] and the two cu_seqlens."""
    lengths_k = lengths_q if lengths_k is None else lengths_k
    Hkv = H if Hkv is None else Hkv
    cq, ck = cu_seqlens(lengths_q), cu_seqlens(lengths_k)
    tq, tk = int(cq[-1]), int(ck[-1])
    q = randn_bf16((tq, H, d), seed * 3 + 0, device)
    k = randn_bf16((tk, Hkv, d), seed * 3 + 1, device)
    v = randn_bf16((tk, Hkv, d), seed * 3 + 2, device)
    return q, k, v, cq.to(device), ck.to(device)


@dataclass
class PagedBatch:
    q: torch.Tensor            # [B, H, d]
    k_cache: torch.Tensor      # [num_pages, 16, Hkv, d]
    v_cache: torch.Tensor
    block_table: torch.Tensor  # int32 [B, max_pages]
    seqlens: torch.Tensor      # int32 [B]
    lengths: list
    max_seqlen: int
    num_pages: int


def paged_inputs(lengths, H, d, seed: int, device="cpu", Hkv=None, page_size=PAGE_SIZE, slack_pages=0,
                 pad_value=-1, pool_on_device=False, max_pages=None, k_signs=False) -> PagedBatch:
    """A page pool holding every sequence's KV, pages assigned by a seeded
    random permutation; unused block_table entries hold ``pad_value``.
    ``k_signs`` draws the key pool as uniform signs instead of N(0, 1)."""
    Hkv = H if Hkv is None else Hkv
    B = len(lengths)
    pages_per = [(L + page_size - 1) // page_size for L in lengths]
    num_pages = max(1, sum(pages_per) + slack_pages)
    perm = torch.randperm(num_pages, generator=_gen(seed * 7 + 5)).to(torch.int32)
    maxp = max(1, max(pages_per)) if max_pages is None else max_pages
    bt = torch.full((B, maxp), pad_value, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(pages_per):
        bt[b, :n] = perm[pos:pos + n]
        pos += n
    shape = (num_pages, page_size, Hkv, d)
    if pool_on_device:
        kc = (sign_bf16_device if k_signs else randn_bf16_device)(shape, seed * 7 + 1, device)
        vc = randn_bf16_device(shape, seed * 7 + 2, device)
    else:
        kc = (sign_bf16 if k_signs else randn_bf16)(shape, seed * 7 + 1, device)
        vc = randn_bf16(shape, seed * 7 + 2, device)
    q = randn_bf16((B, H, d), seed * 7 + 0, device)
    return PagedBatch(q, kc, vc, bt.to(device), torch.tensor(lengths, dtype=torch.int32).to(device),
                      list(lengths), max(lengths) if lengths else 0, num_pages)


def c4_lengths(seed: int = 1238) -> list[int]:
    return uniform_lengths(VARLEN_C4["num_seqs"], VARLEN_C4["lo"], VARLEN_C4["hi"], seed)


def c5_lengths(seed: int = 1239) -> list[int]:
    return uniform_lengths(PAGED_C5["B"], PAGED_C5["lo"], PAGED_C5["hi"], seed)


@dataclass
class ChunkBatch:
    q: torch.Tensor            # [total_q, H, d], the newest tokens of each sequence
    k_cache: torch.Tensor      # [num_pages, 16, Hkv, d]
    v_cache: torch.Tensor
    block_table: torch.Tensor  # int32 [S, max_pages]
    cu_q: torch.Tensor         # int32 [S + 1]
    cu_k: torch.Tensor         # int32 [S + 1]
    lengths_q: list
    lengths_k: list
    max_q: int
    max_k: int
    num_pages: int


def chunk_inputs(lengths_q, lengths_k, H, d, seed: int, device="cpu", Hkv=None, page_size=PAGE_SIZE,
                 slack_pages=0, stale=float("nan"), pool_on_device=False, k_signs=False) -> ChunkBatch:
    """A prefill chunk that continues cached prefixes: sequence s has
    lengths_k[s] keys in the page pool (pages in a seeded random permutation)
    and its lengths_q[s] newest tokens as queries.  Every slot no sequence
    uses (the tail of each last page, the slack pages) holds ``stale``.
    ``k_signs`` draws the key pool as uniform signs instead of N(0, 1)."""
    Hkv = H if Hkv is None else Hkv
    S = len(lengths_k)
    pages_per = [(L + page_size - 1) // page_size for L in lengths_k]
    num_pages = max(1, sum(pages_per) + slack_pages)
    perm = torch.randperm(num_pages, generator=_gen(seed * 11 + 5)).to(torch.int32)
    maxp = max(1, max(pages_per))
    bt = torch.full((S, maxp), -1, dtype=torch.int32)
    used = torch.zeros((num_pages, page_size), dtype=torch.bool)
    pos = 0
    for s, n in enumerate(pages_per):
        bt[s, :n] = perm[pos:pos + n]
        pos += n
        for t in range(0, lengths_k[s], page_size):
            used[int(bt[s, t // page_size]), : min(page_size, lengths_k[s] - t)] = True
    shape = (num_pages, page_size, Hkv, d)
    if pool_on_device:
        kc = (sign_bf16_device if k_signs else randn_bf16_device)(shape, seed * 11 + 1, device)
        vc = randn_bf16_device(shape, seed * 11 + 2, device)
    else:
        kc = (sign_bf16 if k_signs else randn_bf16)(shape, seed * 11 + 1, device)
        vc = randn_bf16(shape, seed * 11 + 2, device)
    if stale is not None:
        mask = (~used).to(kc.device)
        kc[mask] = stale
        vc[mask] = stale
    cq, ck = cu_seqlens(lengths_q), cu_seqlens(lengths_k)
    q = randn_bf16((int(cq[-1]), H, d), seed * 11 + 0, device)
    return ChunkBatch(q, kc, vc, bt.to(device), cq.to(device), ck.to(device), list(lengths_q), list(lengths_k),
                      max(lengths_q), max(lengths_k), num_pages)


def chunk_lengths(seed: int = 1240):
    """(new-token lengths, key lengths) of the continuation workload: key
    length = cached context U[ctx_lo, ctx_hi] + new tokens U[new_lo, new_hi]."""
    ctx = uniform_lengths(CHUNK["num_seqs"], CHUNK["ctx_lo"], CHUNK["ctx_hi"], seed)
    new = uniform_lengths(CHUNK["num_seqs"], CHUNK["new_lo"], CHUNK["new_hi"], seed + 1)
    return new, [c + n for c, n in zip(ctx, new)]
