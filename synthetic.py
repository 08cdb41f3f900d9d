"""Seeded synthetic inputs for the NVFP4 paged-KV tests and benchmark.

This module only draws random data and page tables; it holds none of the NVFP4 arithmetic, so
both the CPU oracle and the GPU library can be fed from it without sharing any of the method.
Every tensor comes from a ``torch.Generator`` seeded explicitly (default seed 0).

Workloads (shapes follow the source pages: 16/32/64-token pages, GQA head_dim 128, contexts of
32K-128K tokens; the pages' own traces and models are not used, these stand in for them):

* ``tiny_decode``    1 sequence of 256 tokens, 8 query / 2 KV heads, head_dim 128, page 16.
* ``page_roundtrip`` 4096 pages x 32 tokens x 8 KV heads x 128, K and V ~ N(0,1) BF16 with 1% of
                     16-value blocks scaled by 1e3 and a disjoint 1% scaled by 1e-3.
* ``decode_batch``   32 sequences x 8192 tokens, 32 query / 8 KV heads, page 64, pool of 4096
                     pages placed by a random permutation.
* ``long_context``   8 sequences with lengths uniform in [32768, 131072], 64 query / 8 KV heads.
* ``extend``         16 sequences with a 4096-token cached prefix (64 pages each) and a
                     512-token BF16 chunk each (8 new pages per sequence).

K carries four outlier channels (13, 42, 77, 118) scaled by 20 in the decode workloads.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

K_OUTLIER_CHANNELS = (13, 42, 77, 118)
K_OUTLIER_FACTOR = 20.0


def gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, g: torch.Generator, device="cpu") -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)


def kv_pages_bf16(num_pages, H, T, D, g, k_outliers=False, device="cpu") -> torch.Tensor:
    """[num_pages, H, T, D] BF16 ~ N(0,1); optionally the K outlier channels x20."""
    x = torch.randn((num_pages, H, T, D), generator=g, dtype=torch.float32, device=device)
    if k_outliers:
        ch = [c for c in K_OUTLIER_CHANNELS if c < D]
        x[..., ch] *= K_OUTLIER_FACTOR
    return x.to(torch.bfloat16)


def outlier_blocks_bf16(num_pages, H, T, D, g, frac_big=0.01, frac_small=0.01,
                        big=1e3, small=1e-3, device="cpu") -> torch.Tensor:
    """N(0,1) pages where exactly frac_big of the 16-value blocks are scaled by `big` and a
    disjoint frac_small of them by `small`, the blocks chosen by a seeded permutation."""
    x = torch.randn((num_pages, H, T, D), generator=g, dtype=torch.float32, device=device)
    blocks = x.view(-1, 16)
    nb = blocks.shape[0]
    n_big, n_small = int(nb * frac_big), int(nb * frac_small)
    perm = torch.randperm(nb, generator=g, device=device)
    blocks[perm[:n_big]] *= big
    blocks[perm[n_big:n_big + n_small]] *= small
    return x.to(torch.bfloat16)


def random_fp8_bytes(shape, g, device="cpu") -> torch.Tensor:
    """Uniformly random finite E4M3 bit patterns (the two NaN codes 0x7F / 0xFF excluded)."""
    b = torch.randint(0, 254, shape, generator=g, dtype=torch.int32, device=device)
    b = b + (b >= 0x7F).to(torch.int32)  # skip 0x7F; 254 values -> 0..0xFE minus 0x7F
    return b.to(torch.uint8)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def fp16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def permuted_page_table(B, pages_per_seq, pool_pages, g, device="cpu") -> torch.Tensor:
    """[B, pages_per_seq] int32: the first B*pages_per_seq entries of a random permutation of
    the pool, so every sequence's pages are scattered over the pool."""
    assert B * pages_per_seq <= pool_pages
    perm = torch.randperm(pool_pages, generator=g, device=device)[:B * pages_per_seq]
    return perm.view(B, pages_per_seq).to(torch.int32)


@dataclass
class DecodeWorkload:
    name: str
    B: int
    Hq: int
    H: int
    D: int
    T: int
    seq_lens: list
    pool_pages: int
    seed: int = 0
    sm_scale: float = field(default=0.0)

    def __post_init__(self):
        if not self.sm_scale:
            self.sm_scale = 1.0 / math.sqrt(self.D)

    @property
    def max_pages(self) -> int:
        return max(1, max((L + self.T - 1) // self.T for L in self.seq_lens))

    @property
    def kv_tokens(self) -> int:
        return int(sum(self.seq_lens))

    def make(self, device="cpu"):
        """Draw (q [B,Hq,D] bf16, k, v [pool,H,T,D] bf16, page_table [B,max_pages] i32,
        seq_lens [B] i32). Unused page-table entries point at page 0 of the pool."""
        g = gen(self.seed, device)
        q = randn_bf16((self.B, self.Hq, self.D), g, device)
        k = kv_pages_bf16(self.pool_pages, self.H, self.T, self.D, g, k_outliers=True,
                          device=device)
        v = kv_pages_bf16(self.pool_pages, self.H, self.T, self.D, g, device=device)
        need = [(L + self.T - 1) // self.T for L in self.seq_lens]
        perm = torch.randperm(self.pool_pages, generator=g, device=device)
        pt = torch.zeros((self.B, self.max_pages), dtype=torch.int32, device=device)
        off = 0
        for b, n in enumerate(need):
            pt[b, :n] = perm[off:off + n].to(torch.int32)
            off += n
        assert off <= self.pool_pages, "pool too small for the sequences"
        sl = torch.tensor(self.seq_lens, dtype=torch.int32, device=device)
        return q, k, v, pt, sl


def tiny_decode(seed=0) -> DecodeWorkload:
    return DecodeWorkload("tiny decode", B=1, Hq=8, H=2, D=128, T=16, seq_lens=[256],
                          pool_pages=16, seed=seed)


def decode_batch(seed=0) -> DecodeWorkload:
    return DecodeWorkload("decode batch", B=32, Hq=32, H=8, D=128, T=64, seq_lens=[8192] * 32,
                          pool_pages=4096, seed=seed)


def long_context_lengths(seed=0, B=8, lo=32768, hi=131072):
    g = gen(seed + 1000)
    return torch.randint(lo, hi + 1, (B,), generator=g).tolist()


def long_context(seed=0) -> DecodeWorkload:
    lens = long_context_lengths(seed)
    T = 64
    pool = sum((L + T - 1) // T for L in lens)
    return DecodeWorkload("long context", B=8, Hq=64, H=8, D=128, T=T, seq_lens=lens,
                          pool_pages=pool, seed=seed)


@dataclass
class RoundTripWorkload:
    name: str = "page round-trip"
    P: int = 4096
    T: int = 32
    H: int = 8
    D: int = 128
    seed: int = 0

    def make(self, device="cpu"):
        g = gen(self.seed, device)
        k = outlier_blocks_bf16(self.P, self.H, self.T, self.D, g, device=device)
        v = outlier_blocks_bf16(self.P, self.H, self.T, self.D, g, device=device)
        return k, v


@dataclass
class ExtendWorkload:
    name: str = "extend"
    B: int = 16
    prefix: int = 4096
    chunk: int = 512
    Hq: int = 32
    H: int = 8
    D: int = 128
    T: int = 64
    seed: int = 0

    @property
    def prefix_pages(self) -> int:
        return self.B * self.prefix // self.T

    @property
    def chunk_pages(self) -> int:
        return self.B * self.chunk // self.T

    def make(self, device="cpu"):
        """(prefix_bf16 [pool,H,T,D] source of the cached prefix, prefix page table
        [B, prefix/T] into a pool of prefix_pages + chunk_pages pages, chunk_bf16
        [chunk_pages,H,T,D], chunk destination page ids [chunk_pages])."""
        g = gen(self.seed, device)
        pool = self.prefix_pages + self.chunk_pages
        prefix = kv_pages_bf16(pool, self.H, self.T, self.D, g, device=device)
        perm = torch.randperm(pool, generator=g, device=device).to(torch.int32)
        pt = perm[:self.prefix_pages].view(self.B, self.prefix // self.T).contiguous()
        chunk_dst = perm[self.prefix_pages:].contiguous()
        chunk = kv_pages_bf16(self.chunk_pages, self.H, self.T, self.D, g, device=device)
        return prefix, pt, chunk, chunk_dst
