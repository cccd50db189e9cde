"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Every draw is fp32 from a seeded ``torch.Generator``
and is then rounded to the target dtype with round-to-nearest-even, so the
oracle and the CUDA path are handed identical bit patterns.

Recipes (one per workload shape used by the library's tests and benchmark):

* forward: Q, K, V drawn in that order, iid N(0, 1) scaled by ``amp`` in fp32,
  shape [B, H, N, d].
* forward with outliers: as above, then a seeded 0.1% of the entries of each
  tensor multiplied by 10 (the pages give no recipe for outlier inputs).
* rotation signs: d iid fair signs, fp32 +-1.
* paged decode: q [S, H, D] ~ N(0,1); k_cache [nb, H, D/x, bs, x] and v_cache
  [nb, H, D, bs] ~ N(0,1); context_lens ~ U{1..max_ctx}; block_tables is a
  random permutation of the nb = S * max_blocks physical blocks, viewed as
  [S, max_blocks] int32.  The cache layouts are the ones of the
  "PagedAttention" page (data-sketchers.com, section "Inputs"), with x the
  number of elements in one 16-byte vector.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


def _randn(shape, gen, device="cpu"):
    return torch.randn(*shape, generator=gen, dtype=torch.float32, device=device)


def forward_inputs(B: int, H: int, N: int, d: int, dtype=torch.bfloat16, seed: int = 0,
                   amp: float = 1.0, device="cpu"):
    """Q, K, V of shape [B, H, N, d], iid N(0,1)*amp, rounded RNE to ``dtype``."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    out = []
    for _ in range(3):
        t = _randn((B, H, N, d), g)
        if amp != 1.0:
            t = t * amp
        out.append(t.to(dtype).to(device))
    return tuple(out)


def grad_output(B: int, H: int, N: int, d: int, dtype=torch.bfloat16, seed: int = 0,
                device="cpu"):
    """An upstream gradient dO of shape [B, H, N, d], iid N(0,1), rounded RNE
    to ``dtype`` (drawn from its own seed stream, distinct from Q, K, V)."""
    g = torch.Generator(device="cpu").manual_seed(seed + 0x5EED)
    return _randn((B, H, N, d), g).to(dtype).to(device)


def outlier_inputs(B: int, H: int, N: int, d: int, dtype=torch.bfloat16, seed: int = 0,
                   frac: float = 1e-3, amp: float = 10.0, device="cpu"):
    """Q, K, V like :func:`forward_inputs`, with a seeded fraction ``frac`` of
    the entries of each scaled by ``amp``: the few large-magnitude values that
    hurt a per-block 8-bit scale."""
    g = torch.Generator(device="cpu").manual_seed(seed + 0x0F7)
    out = []
    for _ in range(3):
        t = _randn((B, H, N, d), g)
        sel = torch.rand((B, H, N, d), generator=g) < frac
        t = torch.where(sel, t * amp, t)
        out.append(t.to(dtype).to(device))
    return tuple(out)


def rotation_signs(d: int, seed: int = 0, device="cpu"):
    """d random signs (+1.0 / -1.0, fp32): the diagonal of the random
    orthogonal transform used before FP8 quantization."""
    g = torch.Generator(device="cpu").manual_seed(seed + 0x51C)
    bits = torch.randint(0, 2, (d,), generator=g)
    return (1.0 - 2.0 * bits.to(torch.float32)).to(device)


def sample_rows(N: int, count: int, seed: int):
    """``count`` distinct query rows in [0, N), seeded, sorted ascending."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    count = min(count, N)
    return torch.sort(torch.randperm(N, generator=g)[:count]).values


@dataclass
class DecodeInputs:
    q: torch.Tensor             # [S, H, D]
    k_cache: torch.Tensor       # [nb, Hk, D/x, bs, x]  (Hk = key/value heads)
    v_cache: torch.Tensor       # [nb, Hk, D, bs]
    block_tables: torch.Tensor  # int32 [S, max_blocks]
    context_lens: torch.Tensor  # int32 [S]
    block_size: int
    scale: float

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def num_kv_heads(self) -> int:
        return int(self.k_cache.shape[1])

    def kv_bytes_read(self) -> int:
        """Algorithmic K and V bytes one decode reads: every context token's key
        and value, once for every key/value head."""
        S, H, D = self.q.shape
        es = self.q.element_size()
        return int(self.context_lens.to(torch.int64).sum().item()) * self.num_kv_heads * D * es * 2


def decode_inputs(num_seqs: int, num_heads: int, head_size: int, block_size: int,
                  max_ctx: int, dtype=torch.bfloat16, seed: int = 0, device="cpu",
                  min_ctx: int = 1, scale: float | None = None,
                  num_kv_heads: int | None = None) -> DecodeInputs:
    """Paged-decode inputs.  The caches are drawn on ``device`` (a seeded CUDA
    generator when it is a GPU, in chunks, so multi-GiB caches never pass
    through host memory); the small tensors always come from a CPU generator.
    ``num_kv_heads`` (default num_heads) sets the caches' key/value head axis."""
    if num_kv_heads is None:
        num_kv_heads = num_heads
    es = torch.tensor([], dtype=dtype).element_size()
    x = 16 // es
    assert head_size % x == 0
    max_blocks = (max_ctx + block_size - 1) // block_size
    nb = num_seqs * max_blocks
    g = torch.Generator(device="cpu").manual_seed(seed)
    q = _randn((num_seqs, num_heads, head_size), g).to(dtype)
    context_lens = torch.randint(min_ctx, max_ctx + 1, (num_seqs,), generator=g,
                                 dtype=torch.int64).to(torch.int32)
    block_tables = torch.randperm(nb, generator=g).view(num_seqs, max_blocks).to(torch.int32)
    dev = torch.device(device)
    gdev = torch.Generator(device=dev).manual_seed(seed + 1000003)
    k_cache = torch.empty((nb, num_kv_heads, head_size // x, block_size, x), dtype=dtype,
                          device=dev)
    v_cache = torch.empty((nb, num_kv_heads, head_size, block_size), dtype=dtype, device=dev)
    chunk = max(1, (1 << 26) // (num_kv_heads * head_size * block_size))  # blocks per chunk
    for cache in (k_cache, v_cache):
        flat = cache.view(nb, -1)
        for b0 in range(0, nb, chunk):
            b1 = min(nb, b0 + chunk)
            flat[b0:b1] = torch.randn((b1 - b0, flat.shape[1]), generator=gdev,
                                      dtype=torch.float32, device=dev).to(dtype)
    if scale is None:
        scale = head_size ** -0.5
    return DecodeInputs(q.to(dev), k_cache, v_cache, block_tables.to(dev),
                        context_lens.to(dev), block_size, float(scale))
