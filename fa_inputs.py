"""Seeded synthetic inputs for the attention forward, shared by the tests, the
bench and the smoke check.

This module holds no attention arithmetic: it only draws random tensors and
sequence lengths.  Both the CUDA path and the float64 oracle consume what it
returns; neither side computes its inputs itself.

Recipe (the pages give no workloads, so these follow the five configurations
this library is measured on):

* every tensor is drawn in fp32 from ``torch.randn`` with a seeded generator,
  multiplied by its standard deviation, then rounded once to the device dtype
  (bf16 round-to-nearest-even, or kept fp32);
* sequence lengths are drawn with ``torch.randint`` from the same generator,
  before any tensor;
* ``device="cpu"`` uses a CPU generator; ``device="cuda"`` uses a CUDA
  generator seeded the same way (a different stream of numbers: only the
  seed is shared).  The very large decode KV cache is drawn on the device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


def _gen(device: str, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn(shape, *, std: float = 1.0, dtype=torch.bfloat16, device="cpu",
          gen: torch.Generator) -> torch.Tensor:
    """fp32 N(0, std^2) draw rounded once to ``dtype``."""
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


@dataclass
class DenseCase:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    scale: float
    causal: bool
    meta: dict = field(default_factory=dict)


@dataclass
class VarlenCase:
    q: torch.Tensor  # [T, H, D]
    k: torch.Tensor
    v: torch.Tensor
    cu_seqlens: torch.Tensor  # int32 [num_seqs + 1], on the CPU
    max_seqlen: int
    scale: float
    causal: bool
    meta: dict = field(default_factory=dict)


@dataclass
class DecodeCase:
    q: torch.Tensor        # [B, H, D]
    k_cache: torch.Tensor  # [T_k, H, D] packed
    v_cache: torch.Tensor
    cu_seqlens_k: torch.Tensor  # int32 [B + 1], on the CPU
    num_splits: int
    scale: float
    meta: dict = field(default_factory=dict)


def dense(B, H, N, D, *, seed, causal, dtype=torch.bfloat16, qk_std=1.0,
          v_std=1.0, scale=None, device="cpu") -> DenseCase:
    g = _gen(device, seed)
    q = randn((B, H, N, D), std=qk_std, dtype=dtype, device=device, gen=g)
    k = randn((B, H, N, D), std=qk_std, dtype=dtype, device=device, gen=g)
    v = randn((B, H, N, D), std=v_std, dtype=dtype, device=device, gen=g)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    return DenseCase(q, k, v, float(scale), bool(causal),
                     dict(B=B, H=H, N=N, D=D, seed=seed, qk_std=qk_std))


def output_grad(shape, *, seed, std=1.0, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """The loss gradient dO fed to the backward: N(0, std^2), rounded once."""
    return randn(shape, std=std, dtype=dtype, device=device, gen=_gen(device, seed))


def stats_rows(R, C, *, seed, loc=0.0, std=1.0, row_spread=0.0, dtype=torch.bfloat16,
               device="cpu") -> torch.Tensor:
    """A [R, C] matrix for the row statistics: row r is loc_r + std * z with
    z ~ N(0, 1) and loc_r = loc + row_spread * g_r, g_r ~ N(0, 1) (drawn
    first), computed in fp32 and rounded once to ``dtype``."""
    g = _gen(device, seed)
    offs = torch.randn((R, 1), generator=g, device=device, dtype=torch.float32)
    x = torch.randn((R, C), generator=g, device=device, dtype=torch.float32)
    x.mul_(std).add_(offs * row_spread + loc)
    return x.to(dtype)


def varlen_lengths(total_tokens: int, max_len: int, *, gen: torch.Generator,
                   min_len: int = 1) -> list[int]:
    """Draw lengths U[min_len, max_len] until they cover ``total_tokens``;
    the last one is cut so that the lengths sum to ``total_tokens`` exactly."""
    lens: list[int] = []
    s = 0
    while s < total_tokens:
        n = int(torch.randint(min_len, max_len + 1, (1,), generator=gen).item())
        n = min(n, total_tokens - s)
        lens.append(n)
        s += n
    return lens


def cu_from_lengths(lens) -> torch.Tensor:
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def varlen(lens=None, *, H, D, seed, causal=True, total_tokens=None,
           max_len=None, dtype=torch.bfloat16, scale=None,
           device="cpu") -> VarlenCase:
    """Packed [T, H, D] inputs.  Either give ``lens`` or (``total_tokens``,
    ``max_len``) to draw them."""
    g = _gen("cpu", seed)
    if lens is None:
        lens = varlen_lengths(total_tokens, max_len, gen=g)
    lens = [int(n) for n in lens]
    T = sum(lens)
    gd = g if device == "cpu" else _gen(device, seed)
    q = randn((T, H, D), dtype=dtype, device=device, gen=gd)
    k = randn((T, H, D), dtype=dtype, device=device, gen=gd)
    v = randn((T, H, D), dtype=dtype, device=device, gen=gd)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    return VarlenCase(q, k, v, cu_from_lengths(lens), max(lens) if lens else 0,
                      float(scale), bool(causal),
                      dict(H=H, D=D, seed=seed, lens=lens, T=T))


def decode(B, H, D, *, seed, num_splits, lens=None, min_len=1024,
           max_len=32768, dtype=torch.bfloat16, scale=None,
           device="cpu") -> DecodeCase:
    """One query token per sequence; a packed KV cache of ``sum(lens)`` rows.
    Lengths are drawn on the CPU generator first, the tensors after."""
    g = _gen("cpu", seed)
    if lens is None:
        lens = [int(x) for x in
                torch.randint(min_len, max_len + 1, (B,), generator=g).tolist()]
    lens = [int(n) for n in lens]
    assert len(lens) == B
    T = sum(lens)
    gd = g if device == "cpu" else _gen(device, seed)
    q = randn((B, H, D), dtype=dtype, device=device, gen=gd)
    kc = randn((T, H, D), dtype=dtype, device=device, gen=gd)
    vc = randn((T, H, D), dtype=dtype, device=device, gen=gd)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    return DecodeCase(q, kc, vc, cu_from_lengths(lens), int(num_splits),
                      float(scale), dict(B=B, H=H, D=D, seed=seed, lens=lens,
                                         T=T))


@dataclass
class PagedDecodeCase:
    q: torch.Tensor            # [B, H, D]
    k_pages: torch.Tensor      # [num_pages, page_size, H_kv, D]
    v_pages: torch.Tensor
    block_table: torch.Tensor  # int32 [B, max_blocks], on the CPU
    seqlens: torch.Tensor      # int32 [B], on the CPU
    num_splits: int
    scale: float
    meta: dict = field(default_factory=dict)


def paged_decode(B, H, H_kv, D, page_size, *, seed, num_splits, lens=None,
                 min_len=1024, max_len=32768, spare_pages=3, dtype=torch.bfloat16,
                 scale=None, device="cpu") -> PagedDecodeCase:
    """A paged KV cache: every sequence gets ceil(L / page_size) pages drawn
    without replacement (a seeded permutation) from a pool with a few spare
    pages; unused block-table entries are -1.  Lengths are drawn first, on the
    CPU generator, exactly as in ``decode``."""
    g = _gen("cpu", seed)
    if lens is None:
        lens = [int(x) for x in
                torch.randint(min_len, max_len + 1, (B,), generator=g).tolist()]
    lens = [int(n) for n in lens]
    nblk = [-(-L // page_size) for L in lens]
    P = sum(nblk) + spare_pages
    perm = torch.randperm(P, generator=g).tolist()
    table = torch.full((B, max(1, max(nblk) if nblk else 1)), -1, dtype=torch.int32)
    i = 0
    for b in range(B):
        for c in range(nblk[b]):
            table[b, c] = perm[i]
            i += 1
    gd = g if device == "cpu" else _gen(device, seed)
    q = randn((B, H, D), dtype=dtype, device=device, gen=gd)
    kp = randn((P, page_size, H_kv, D), dtype=dtype, device=device, gen=gd)
    vp = randn((P, page_size, H_kv, D), dtype=dtype, device=device, gen=gd)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    return PagedDecodeCase(q, kp, vp, table, torch.tensor(lens, dtype=torch.int32),
                           int(num_splits), float(scale),
                           dict(B=B, H=H, H_kv=H_kv, D=D, page_size=page_size,
                                seed=seed, lens=lens, pages=P))


# The five measured configurations, by number.
def config1(device="cpu") -> DenseCase:
    """B=1 H=1 N=256 D=64, fp32 N(0,1), scale 1/8, non-causal."""
    return dense(1, 1, 256, 64, seed=1, causal=False, dtype=torch.float32,
                 device=device)


def config2(device="cpu") -> DenseCase:
    """B=4 H=16 N=2048 D=128, bf16 N(0,1), causal."""
    return dense(4, 16, 2048, 128, seed=2, causal=True, device=device)


def config3(device="cpu") -> DenseCase:
    """B=1 H=32 N=16384 D=128, bf16, causal; Q,K ~ N(0, 3^2), V ~ N(0,1):
    scaled scores have std ~9 and reach the high tens (overflow stress)."""
    return dense(1, 32, 16384, 128, seed=3, causal=True, qk_std=3.0,
                 device=device)


def config4(device="cpu") -> DecodeCase:
    """Split-KV decode: B=64 H=32 D=128, KV lengths U[1024, 32768], 16 chunks."""
    return decode(64, 32, 128, seed=4, num_splits=16, device=device)


def config5(D: int, device="cpu") -> VarlenCase:
    """Ragged varlen prefill: 65536 tokens, lengths U[1, 8192], H=16, causal."""
    return varlen(H=16, D=D, seed=5, causal=True, total_tokens=65536,
                  max_len=8192, device=device)
