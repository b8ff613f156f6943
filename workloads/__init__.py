"""Seeded synthetic inputs for paged MLA decode.

This module is the only code shared by the CUDA path's tests/bench and the
CPU oracle.  It draws random numbers and lays out a paged cache; it holds
none of the attention arithmetic.

Layouts follow the FlashMLA-PyTorch interface page (``flash_mla_interface.py``,
docstring of ``flash_mla_with_kvcache``):

* ``q``            (batch, s_q, h_q, 576) bf16 -- 512 latent dims + 64 RoPE dims
* ``k_cache``      (num_blocks, 64, h_k, 576) bf16 -- the first 512 dims are V
* ``block_table``  (batch, max_blocks_per_seq) int32, logical block -> physical
                   block, padded with -1 past ``ceil(L/64)``
* ``cache_seqlens`` (batch,) int32

Workloads (sizes from the DeepSeek-V3-shaped decode settings, all synthetic):

====================  ====  ===  ===  =====================================
name                  B     s_q  h_q  cache_seqlens
====================  ====  ===  ===  =====================================
tiny                  2     1    16   {100, 257}, 8-block pool, one unused
dsv3_decode           64    1    128  i.i.d. U{1..8192}
mtp_causal            128   2    128  all 4096, causal
skewed_long           32    1    128  [131072] + [1024] * 31
lowhead_tp            256   1    16   i.i.d. U{2048..16384}, q ~ 0.5 N(0,1)
====================  ====  ===  ===  =====================================

Physical blocks are a seeded random permutation of a pool sized to the
sum of blocks (``randperm(pool)`` handed out in order).  For parity runs the
unused tail rows of every last page and every unused physical block are
filled with NaN, so that any read past ``cache_seqlens`` shows up in the
output; timing runs fill them with N(0,1) instead.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional, Sequence

import torch

PAGE = 64
D_QK = 576
D_V = 512


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    s_q: int
    h_q: int
    h_k: int = 1
    causal: bool = False
    # one of: ("fixed", [L...]), ("uniform", lo, hi), ("long_plus", long, short)
    seqlens: tuple = ("fixed", (1,))
    q_std: float = 1.0
    k_std: float = 1.0
    extra_pool_blocks: int = 0
    description: str = ""

    @property
    def rows(self) -> int:
        """Query rows per KV head: s_q * h_q / h_k (num_heads_per_head_k)."""
        return self.s_q * self.h_q // self.h_k

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload(
        "tiny", batch=2, s_q=1, h_q=16, seqlens=("fixed", (100, 257)),
        extra_pool_blocks=1,
        description="batch=2 s_q=1 h_q=16 L={100,257}, 8-block pool"),
    "dsv3_decode": Workload(
        "dsv3_decode", batch=64, s_q=1, h_q=128, seqlens=("uniform", 1, 8192),
        description="DeepSeek-V3-shaped decode: batch=64 s_q=1 h_q=128 L~U[1,8192]"),
    "mtp_causal": Workload(
        "mtp_causal", batch=128, s_q=2, h_q=128, causal=True,
        seqlens=("fixed", (4096,)),
        description="MTP/speculative decode: batch=128 s_q=2 h_q=128 L=4096 causal"),
    "skewed_long": Workload(
        "skewed_long", batch=32, s_q=1, h_q=128,
        seqlens=("long_plus", 131072, 1024),
        description="skewed long context: batch=32 L=[131072, 1024 x 31]"),
    "lowhead_tp": Workload(
        "lowhead_tp", batch=256, s_q=1, h_q=16, seqlens=("uniform", 2048, 16384),
        q_std=0.5,
        description="TP-sliced low-head decode: batch=256 h_q=16 L~U[2048,16384]"),
}

# Order in which the workloads are listed (the second one is the headline).
WORKLOAD_ORDER = ["tiny", "dsv3_decode", "mtp_causal", "skewed_long", "lowhead_tp"]
DEFAULT_SEED_BASE = 1234


def seed_for(name: str) -> int:
    return DEFAULT_SEED_BASE + WORKLOAD_ORDER.index(name) if name in WORKLOAD_ORDER \
        else DEFAULT_SEED_BASE + 97


def draw_seqlens(w: Workload, gen: torch.Generator) -> torch.Tensor:
    kind = w.seqlens[0]
    if kind == "fixed":
        vals = list(w.seqlens[1])
        if len(vals) == 1:
            vals = vals * w.batch
        assert len(vals) == w.batch
        return torch.tensor(vals, dtype=torch.int32)
    if kind == "uniform":
        lo, hi = w.seqlens[1], w.seqlens[2]
        return torch.randint(lo, hi + 1, (w.batch,), generator=gen, dtype=torch.int64).to(torch.int32)
    if kind == "long_plus":
        return torch.tensor([w.seqlens[1]] + [w.seqlens[2]] * (w.batch - 1), dtype=torch.int32)
    raise ValueError(kind)


@dataclass
class Inputs:
    workload: Workload
    q: torch.Tensor
    k_cache: torch.Tensor
    block_table: torch.Tensor
    cache_seqlens: torch.Tensor
    scale: float
    seed: int
    extra: dict = field(default_factory=dict)

    @property
    def num_blocks(self) -> int:
        return self.k_cache.shape[0]

    def to(self, device) -> "Inputs":
        return Inputs(self.workload, self.q.to(device), self.k_cache.to(device),
                      self.block_table.to(device), self.cache_seqlens.to(device),
                      self.scale, self.seed, dict(self.extra))


def _fill_normal_bf16(t: torch.Tensor, std: float, gen: torch.Generator, chunk: int = 1 << 24):
    """Fill a bf16 tensor with std*N(0,1) in chunks (bounded fp32 scratch)."""
    flat = t.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        tmp = torch.randn(e - s, generator=gen, device=t.device, dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        flat[s:e].copy_(tmp)


def make_inputs(w: Workload | str, seed: Optional[int] = None, device="cpu",
                poison: bool = True, seqlens: Optional[Sequence[int]] = None,
                scale: Optional[float] = None) -> Inputs:
    """Build one seeded input set.

    ``seqlens`` overrides the workload's recipe (used for edge cases).
    Random draws happen on ``device`` with a generator seeded by ``seed``;
    the block permutation and sequence lengths are always drawn on the CPU so
    that they are identical for every device.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    if seed is None:
        seed = seed_for(w.name)
    cpu_gen = torch.Generator(device="cpu").manual_seed(seed)
    if seqlens is not None:
        L = torch.tensor(list(seqlens), dtype=torch.int32)
        w = w.with_(batch=len(L))
    else:
        L = draw_seqlens(w, cpu_gen)
    nblk = [(int(x) + PAGE - 1) // PAGE for x in L.tolist()]
    pool = sum(nblk) + w.extra_pool_blocks
    pool = max(pool, 1)
    perm = torch.randperm(pool, generator=cpu_gen)
    max_blocks = max(max(nblk) if nblk else 0, 1)
    bt = torch.full((w.batch, max_blocks), -1, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = perm[pos:pos + n].to(torch.int32)
        pos += n

    dev_gen = torch.Generator(device=device).manual_seed(seed + 7919)
    q = torch.empty((w.batch, w.s_q, w.h_q, D_QK), dtype=torch.bfloat16, device=device)
    k = torch.empty((pool, PAGE, w.h_k, D_QK), dtype=torch.bfloat16, device=device)
    _fill_normal_bf16(q, w.q_std, dev_gen)
    _fill_normal_bf16(k, w.k_std, dev_gen)
    if poison:
        poison_unused(k, bt, L)
    if scale is None:
        scale = 1.0 / math.sqrt(D_QK)
    return Inputs(w, q, k, bt.to(device), L.to(device), scale, seed)


def e4m3_codes(t: torch.Tensor, chunk: int = 1 << 24) -> torch.Tensor:
    """The e4m3 codes (uint8, same shape and device) of a bf16 input tensor,
    rounded by torch's float8_e4m3fn conversion; NaN stays NaN (0x7f).  Used
    to draw e4m3 query and cache inputs from the seeded bf16 ones."""
    out = torch.empty(t.shape, dtype=torch.uint8, device=t.device)
    src, dst = t.reshape(-1), out.view(-1)
    for s in range(0, src.numel(), chunk):
        e = min(src.numel(), s + chunk)
        dst[s:e] = src[s:e].float().to(torch.float8_e4m3fn).view(torch.uint8)
    return out


def poison_unused(k_cache: torch.Tensor, block_table: torch.Tensor, seqlens: torch.Tensor):
    """Write NaN into every cache row that no sequence may read."""
    bt = block_table.cpu()
    L = seqlens.cpu().tolist()
    used = torch.zeros(k_cache.shape[0], dtype=torch.bool)
    for b, l in enumerate(L):
        n = (l + PAGE - 1) // PAGE
        if n == 0:
            continue
        phys = bt[b, :n].long()
        used[phys] = True
        tail = l - (n - 1) * PAGE
        if tail < PAGE:
            k_cache[int(phys[-1]), tail:] = float("nan")
    unused = (~used).nonzero().flatten()
    if unused.numel():
        k_cache[unused.to(k_cache.device)] = float("nan")


def seqlens_blocks(seqlens) -> list:
    return [(int(x) + PAGE - 1) // PAGE for x in list(seqlens)]
