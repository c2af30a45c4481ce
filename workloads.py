"""Seeded synthetic inputs for the QuantMLA decode path.

This module holds no quantization or attention arithmetic: it only draws
random tensors with the shapes and value distributions of the workloads, so
that the CUDA library and the CPU oracle can be fed identical inputs.

Distributions (the same for every workload):
  * content latent c: N(0, 1) bf16, with 8 channels (drawn once per cache)
    multiplied by 10 -- outlier channels of an MLA latent;
  * RoPE key k_r: N(0, 1) bf16, each frequency pair (2i, 2i+1) multiplied by
    a per-cache factor 10^U(-1, 1);
  * queries q_lat, q_rope: N(0, 1) bf16;
  * page table: the pages a sequence needs, drawn from a random permutation
    of the page pool (64-token pages);
  * softmax scale 1/sqrt(192).
"""

from __future__ import annotations

import dataclasses
import math

import torch

PAGE_TOKENS = 64
D_LATENT = 512
D_ROPE = 64
SOFTMAX_SCALE = 1.0 / math.sqrt(192.0)


@dataclasses.dataclass
class Workload:
    name: str
    mode: str            # "C4R4" | "C2R4" | "BF16"
    B: int
    H: int
    seq_lens: list       # tokens per sequence at decode time
    seed: int
    steps: int = 0       # serving loop: decode steps, each appending one token
    description: str = ""

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seq_lens))


def _uniform_ints(lo: int, hi: int, n: int, seed: int):
    g = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def workload(name: str) -> Workload:
    """The named workloads. Sizes follow the DeepSeek-V2-Lite / V3 MLA shapes."""
    if name == "tiny_c4r4":
        return Workload(name, "C4R4", 2, 16, [1024, 1024], 0,
                        description="B=2, L=1024, H=16, C4R4")
    if name.startswith("v2lite"):
        mode = name.split("_")[1].upper() if "_" in name else "C4R4"
        return Workload(name, mode, 32, 16, _uniform_ints(1024, 32768, 32, 1), 1,
                        description="DeepSeek-V2-Lite-shaped decode: B=32, L~U[1K,32K], H=16, %s" % mode)
    if name.startswith("v3"):
        mode = name.split("_")[1].upper() if "_" in name else "C4R4"
        return Workload(name, mode, 64, 128, [8192] * 64, 2,
                        description="DeepSeek-V3-shaped decode: B=64, L=8192, H=128, %s" % mode)
    if name.startswith("long"):
        mode = name.split("_")[1].upper()
        return Workload(name, mode, 4, 128, [131072] * 4, 3,
                        description="long-context decode: B=4, L=131072, H=128, %s" % mode)
    if name == "serving_c4r4":
        return Workload(name, "C4R4", 128, 16, _uniform_ints(2048, 16384, 128, 4), 4, steps=256,
                        description="serving loop: B=128, H=16, L0~U[2K,16K], 256 append+decode steps")
    raise KeyError(name)


class CacheStats:
    """Per-cache structure of the value distributions (outliers, pair scales)."""

    def __init__(self, seed: int):
        g = torch.Generator().manual_seed(seed * 7919 + 17)
        self.outlier_channels = torch.randperm(D_LATENT, generator=g)[:8].sort().values
        expo = torch.rand(D_ROPE // 2, generator=g) * 2.0 - 1.0
        self.rope_pair_scale = torch.pow(10.0, expo).repeat_interleave(2)   # [64]
        self.latent_scale = torch.ones(D_LATENT)
        self.latent_scale[self.outlier_channels] = 10.0


def make_tokens(n: int, stats: CacheStats, gen: torch.Generator, device="cpu"):
    """n cache tokens: (c_latent bf16 [n,512], k_rope bf16 [n,64])."""
    c = torch.randn(n, D_LATENT, generator=gen, device=device) * stats.latent_scale.to(device)
    k = torch.randn(n, D_ROPE, generator=gen, device=device) * stats.rope_pair_scale.to(device)
    return c.to(torch.bfloat16), k.to(torch.bfloat16)


def make_queries(B: int, H: int, gen: torch.Generator, device="cpu"):
    ql = torch.randn(B, H, D_LATENT, generator=gen, device=device).to(torch.bfloat16)
    qr = torch.randn(B, H, D_ROPE, generator=gen, device=device).to(torch.bfloat16)
    return ql, qr


def make_page_table(capacity_tokens, seed: int, extra_pages: int = 0):
    """Random page allocation. capacity_tokens[b] = tokens sequence b may hold.

    Returns (page_table int32 [B, max_pages] with -1 in unused entries,
    num_pages). Pages are a random permutation of a pool sized to the demand
    plus ``extra_pages`` never-referenced pages.
    """
    need = [max(1, math.ceil(c / PAGE_TOKENS)) for c in capacity_tokens]
    total = sum(need) + extra_pages
    g = torch.Generator().manual_seed(seed * 104729 + 3)
    perm = torch.randperm(total, generator=g).to(torch.int32)
    max_pages = max(need)
    pt = torch.full((len(need), max_pages), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(need):
        pt[b, :n] = perm[off:off + n]
        off += n
    return pt, total


def make_sequences(seq_lens, stats: CacheStats, gen: torch.Generator, device="cpu"):
    """Tokens for every sequence, packed back to back, plus cu offsets [B+1]."""
    total = int(sum(seq_lens))
    c, k = make_tokens(total, stats, gen, device)
    cu = torch.zeros(len(seq_lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(seq_lens, dtype=torch.int64), 0).to(torch.int32)
    return c, k, cu


def generator(seed: int, device="cpu") -> torch.Generator:
    return torch.Generator(device=device).manual_seed(seed)
