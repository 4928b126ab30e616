"""Seeded synthetic inputs for the INT4 KV-cache workloads.

Shared by the tests, the benchmark and the oracle's callers.  This module holds
no arithmetic of the method itself (no quantization, no attention): only the
random inputs, their shapes and the paging of positions onto pages.

Random numbers: a counter-based generator.  Element i of stream ``seed`` is
SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) applied to ``seed * 2^32 + i`` spaced by the golden
gamma 0x9E3779B97F4A7C15; two consecutive outputs give one standard normal by
the Box-Muller transform.  The same function runs on CPU or GPU tensors, so a
test can build its inputs on either device (the bytes handed to both sides of a
parity check are always one and the same tensor).

Workloads (every input fp16 from N(0,1); K gets 4 outlier channels per KV head
scaled x20 before the fp16 rounding; seeds K=1, V=2, q=3, page permutation=4,
ragged lengths=5, outlier channels=6; page size 16; K grouped at 64 and V at
128 unless a group sweep says otherwise).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

SEED_K, SEED_V, SEED_Q, SEED_PERM, SEED_LENS, SEED_OUTLIER, SEED_NEW = 1, 2, 3, 4, 5, 6, 7

_GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB


def _s64(x: int) -> int:
    """A 64-bit constant as the signed int64 torch stores."""
    x &= (1 << 64) - 1
    return x - (1 << 64) if x >= (1 << 63) else x


def _lsr(z: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (z >> k) & ((1 << (64 - k)) - 1)


def splitmix64(seed: int, start: int, n: int, device="cpu") -> torch.Tensor:
    """Outputs start .. start+n-1 of stream ``seed`` as int64 bit patterns."""
    i = torch.arange(start, start + n, dtype=torch.int64, device=device)
    z = (i + 1) * _s64(_GAMMA) + _s64(seed << 32)
    z = (z ^ _lsr(z, 30)) * _s64(_M1)
    z = (z ^ _lsr(z, 27)) * _s64(_M2)
    return z ^ _lsr(z, 31)


def uniform01(seed: int, start: int, n: int, device="cpu") -> torch.Tensor:
    """float64 uniforms in [0, 1) from the top 53 bits."""
    return _lsr(splitmix64(seed, start, n, device), 11).to(torch.float64) * (2.0 ** -53)


def normal(seed: int, n: int, device="cpu") -> torch.Tensor:
    """n standard normals (float32), element j from counters 2j and 2j+1."""
    return _normal_range(seed, 0, n, device)


def randint_below(seed: int, n: int, bound: int, device="cpu") -> torch.Tensor:
    """n integers in [0, bound) (bound small; modulo bias below 2^-40)."""
    return torch.remainder(_lsr(splitmix64(seed, 0, n, device), 11), bound)


def outlier_channels(num_kv_heads: int, head_dim: int, per_head: int = 4, seed: int = SEED_OUTLIER) -> torch.Tensor:
    """[Hkv, per_head] distinct channel indices per KV head (fixed across tokens)."""
    out = torch.empty(num_kv_heads, per_head, dtype=torch.int64)
    draws = randint_below(seed, num_kv_heads * head_dim * 8, head_dim).tolist()
    it = iter(draws)
    for h in range(num_kv_heads):
        chosen: list[int] = []
        while len(chosen) < per_head:
            c = next(it)
            if c not in chosen:
                chosen.append(c)
        out[h] = torch.tensor(chosen)
    return out


def kv_tensor(seed: int, shape: tuple[int, int, int, int], outlier_scale: float = 0.0,
              outlier_idx: torch.Tensor | None = None, device="cpu", token_offset: int = 0) -> torch.Tensor:
    """fp16 [B, n, Hkv, d] from N(0,1); with outliers, channels outlier_idx[h] scaled before rounding.

    Element (b, t, h, i) is counter-indexed by its flat position in a [B, n, Hkv, d]
    array, shifted by ``token_offset`` tokens, so a slice of a long sequence can be
    regenerated on its own.
    """
    B, n, H, d = shape
    x = torch.empty(shape, dtype=torch.float16, device=device)
    per_b = n * H * d
    for b in range(B):
        base = (b * 1_000_003 + token_offset) * H * d  # sequences use disjoint counter ranges
        vals = _normal_range(seed, base, per_b, device).view(n, H, d)
        if outlier_scale and outlier_idx is not None:
            scale = torch.ones(H, d, dtype=torch.float32, device=device)
            scale.scatter_(1, outlier_idx.to(device), outlier_scale)
            vals = vals * scale
        x[b] = vals.to(torch.float16)
    return x


def _normal_range(seed: int, start: int, n: int, device, chunk: int = 1 << 24) -> torch.Tensor:
    out = torch.empty(n, dtype=torch.float32, device=device)
    for s in range(0, n, chunk):
        m = min(chunk, n - s)
        u = uniform01(seed, 2 * (start + s), 2 * m, device).view(m, 2)
        r = torch.sqrt(-2.0 * torch.log(1.0 - u[:, 0]))
        out[s:s + m] = (r * torch.cos((2.0 * math.pi) * u[:, 1])).to(torch.float32)
    return out


def permutation(seed: int, n: int) -> torch.Tensor:
    """A seeded permutation of range(n) (sort by random keys)."""
    keys = splitmix64(seed, 0, n)
    return torch.argsort(keys, stable=True).to(torch.int32)


@dataclass
class Workload:
    """One decode workload: geometry, lengths and paging."""

    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    ctx: list[int]              # cached tokens per sequence before the appended one
    P: int = 16
    Gk: int = 64
    Gv: int = 128
    permute_pages: bool = True
    extra_pages: int = 0
    description: str = ""
    seq_lens: list[int] = field(init=False)

    def __post_init__(self):
        self.seq_lens = [c + 1 for c in self.ctx]  # the appended token is attended to

    @property
    def r(self) -> int:
        return self.Hq // self.Hkv

    @property
    def pages_per_seq(self) -> list[int]:
        return [(L + self.P - 1) // self.P for L in self.seq_lens]

    @property
    def max_blocks(self) -> int:
        return max(self.pages_per_seq)

    @property
    def num_pages(self) -> int:
        return sum(self.pages_per_seq) + self.extra_pages

    @property
    def max_len(self) -> int:
        return max(self.seq_lens)

    def block_table(self) -> torch.Tensor:
        """int32 [B, max_blocks]; unused entries are -1.  Pages are a seeded permutation of the pool."""
        order = permutation(SEED_PERM, self.num_pages) if self.permute_pages else \
            torch.arange(self.num_pages, dtype=torch.int32)
        bt = torch.full((self.B, self.max_blocks), -1, dtype=torch.int32)
        k = 0
        for b, npg in enumerate(self.pages_per_seq):
            bt[b, :npg] = order[k:k + npg]
            k += npg
        return bt

    def with_groups(self, G: int) -> "Workload":
        w = Workload(self.name + f"_g{G}", self.B, self.Hq, self.Hkv, self.d, list(self.ctx), self.P, G, G,
                     self.permute_pages, self.extra_pages, self.description)
        return w

    def packed_bytes_per_token_head(self) -> int:
        """Bytes of packed K+V codes and fp16 scales one token of one KV head occupies."""
        return self.d + 2 * (self.d // self.Gk + self.d // self.Gv)

    def decode_bytes(self) -> int:
        """Algorithmic HBM bytes of one decode attention pass: the packed cache it must read."""
        return self.Hkv * sum(self.seq_lens) * self.packed_bytes_per_token_head()

    def append_bytes(self) -> int:
        """Algorithmic bytes of appending one token per sequence: fp16 K and V read, packed rows written."""
        return self.B * self.Hkv * (2 * self.d * 2 + self.packed_bytes_per_token_head())


def ragged_lengths(B: int, lo: int, hi: int, seed: int = SEED_LENS) -> list[int]:
    return [lo + int(x) for x in randint_below(seed, B, hi - lo + 1).tolist()]


def tiny_mha() -> Workload:
    return Workload("tiny_mha_b1_h8_l512", 1, 8, 8, 128, [512], permute_pages=False,
                    description="1 layer, batch 1, 8 query heads = 8 KV heads, head_dim 128, context 512, "
                                "contiguous 16-token pages")


def llama7b_mha() -> Workload:
    return Workload("llama7b_mha_b8_h32_l8192", 8, 32, 32, 128, [8192] * 8,
                    description="batch 8, 32 query heads = 32 KV heads, head_dim 128, context 8192, "
                                "permuted 16-token pages")


def gqa8b() -> Workload:
    return Workload("gqa8b_b4_h32kv8_l32768", 4, 32, 8, 128, [32768] * 4,
                    description="batch 4, 32 query heads sharing 8 KV heads, head_dim 128, context 32768")


def ragged() -> Workload:
    return Workload("ragged_b32_h32kv8_l512_4096", 32, 32, 8, 128, ragged_lengths(32, 512, 4096),
                    description="batch 32, 32/8 heads, context lengths uniform in [512, 4096] (seed 5), "
                                "shared permuted page pool")


def longctx(G: int = 64) -> Workload:
    """K and V both grouped at G (the group-size sweep)."""
    w = Workload("longctx_b1_h32kv8_l131072", 1, 32, 8, 128, [131072],
                 description="batch 1, 32/8 heads, context 131072, K and V grouped at G")
    return w.with_groups(G)


ALL = {
    "tiny": tiny_mha,
    "llama7b": llama7b_mha,
    "gqa8b": gqa8b,
    "ragged": ragged,
    "longctx": longctx,
}
