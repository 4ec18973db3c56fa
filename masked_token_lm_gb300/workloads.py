"""Seeded synthetic workloads for mask-only logits.

This module only draws inputs: hidden states ``H[L_tot, d]``, the LM-head weight ``W[V, d]`` and
the masked positions (a flat index list, or per-sequence CSR offsets with local indices). It holds
none of the method's arithmetic; both the CUDA path and the CPU oracle take their inputs from here.

Shapes and structure follow the models the pages measure ("Mosaic: Unlocking Long-Context
Inference for Diffusion LLMs via Global Memory", paper review, section 6 "实验结果", LLaDA-8B and
Dream-7B; the dLLM-Serve article "扩散大语言模型内存优化：从理论到系统设计", section 2.2, gives
LLaDA-8B's vocabulary V = 126,464). No weights or datasets are used: H ~ N(0, 1) and
W ~ N(0, 0.02), drawn in fp32 and rounded to bf16 (round-to-nearest-even).

Mask positions: a mask ratio r_m selects M = floor(r_m * L + 1/2) positions drawn uniformly
without replacement and sorted ascending.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch


def mask_count(r_m: float, L: int) -> int:
    """Number of masked positions for ratio ``r_m`` over ``L`` tokens (round half up)."""
    return int(math.floor(r_m * L + 0.5))


def _cpu_gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def make_hidden(L_tot: int, d: int, seed: int, device="cpu") -> torch.Tensor:
    """bf16 hidden states [L_tot, d], N(0, 1)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn((L_tot, d), generator=g, device=device, dtype=torch.float32)
    return x.to(torch.bfloat16)


def make_weight(V: int, d: int, seed: int, device="cpu") -> torch.Tensor:
    """bf16 LM-head weight [V, d], N(0, 0.02)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn((V, d), generator=g, device=device, dtype=torch.float32)
    x.mul_(0.02)
    return x.to(torch.bfloat16)


def uniform_positions(L: int, M: int, seed: int) -> torch.Tensor:
    """M distinct positions in [0, L), uniform without replacement, sorted; int32 (CPU)."""
    if M > L:
        raise ValueError("M > L")
    p = torch.randperm(L, generator=_cpu_gen(seed))[:M]
    return torch.sort(p).values.to(torch.int32)


@dataclasses.dataclass
class MaskSet:
    """Masked positions of one batch.

    ``idx`` is int32 [M]. With ``mask_offsets is None`` it holds global row numbers of ``H``.
    Otherwise sequence ``b`` owns ``idx[mask_offsets[b]:mask_offsets[b+1]]``, whose values are
    positions local to that sequence, and its rows start at ``seq_offsets[b]`` in ``H``.
    """

    idx: torch.Tensor
    seq_offsets: Optional[torch.Tensor] = None
    mask_offsets: Optional[torch.Tensor] = None

    @property
    def M(self) -> int:
        return int(self.idx.numel())

    @property
    def B(self) -> int:
        return 0 if self.mask_offsets is None else int(self.mask_offsets.numel()) - 1

    def to(self, device) -> "MaskSet":
        f = lambda t: None if t is None else t.to(device)
        return MaskSet(f(self.idx), f(self.seq_offsets), f(self.mask_offsets))


def flat_mask(L: int, r_m: float, seed: int) -> MaskSet:
    """One sequence, ratio r_m, uniform positions, sorted."""
    return MaskSet(uniform_positions(L, mask_count(r_m, L), seed))


def block_decode_mask(B: int, L: int, block: int, seed: int) -> MaskSet:
    """B sequences of length L; in each, one contiguous block of ``block`` positions starting at
    a seeded uniform offset in [0, L - block] is masked. CSR offsets, local indices."""
    g = _cpu_gen(seed)
    offs = torch.randint(0, L - block + 1, (B,), generator=g)
    idx = torch.cat([torch.arange(int(o), int(o) + block) for o in offs]).to(torch.int32)
    mask_offsets = (torch.arange(B + 1) * block).to(torch.int32)
    seq_offsets = (torch.arange(B + 1) * L).to(torch.int32)
    return MaskSet(idx, seq_offsets, mask_offsets)


def ragged_mask(B: int, L: int, seed: int) -> MaskSet:
    """B sequences of length L; sequence b draws its own ratio r_b ~ U(0, 1) and masks
    M_b = floor(r_b * L + 1/2) uniform positions (sorted, local). CSR offsets."""
    g = _cpu_gen(seed)
    ratios = torch.rand((B,), generator=g, dtype=torch.float64)
    parts: List[torch.Tensor] = []
    counts = []
    for b in range(B):
        Mb = mask_count(float(ratios[b]), L)
        p = torch.randperm(L, generator=g)[:Mb]
        parts.append(torch.sort(p).values)
        counts.append(Mb)
    idx = torch.cat(parts).to(torch.int32) if parts else torch.zeros(0, dtype=torch.int32)
    mask_offsets = torch.tensor([0] + list(torch.tensor(counts).cumsum(0).tolist()), dtype=torch.int32)
    seq_offsets = (torch.arange(B + 1) * L).to(torch.int32)
    return MaskSet(idx, seq_offsets, mask_offsets)


@dataclasses.dataclass
class Workload:
    """One synthetic batch shape: B sequences of length L (L_tot = B*L rows of H)."""

    name: str
    B: int
    L: int
    d: int
    V: int
    out_dtype: str  # "bf16" or "f32"
    chunk_rows: int  # 0: unchunked
    mask_kind: str  # "flat", "block", "ragged"
    r_m: float = 0.0
    block: int = 0
    seed: int = 1000

    @property
    def L_tot(self) -> int:
        return self.B * self.L

    def mask(self) -> MaskSet:
        if self.mask_kind == "flat":
            return flat_mask(self.L, self.r_m, self.seed + 7)
        if self.mask_kind == "block":
            return block_decode_mask(self.B, self.L, self.block, self.seed + 7)
        if self.mask_kind == "ragged":
            return ragged_mask(self.B, self.L, self.seed + 7)
        raise ValueError(self.mask_kind)

    def hidden(self, device="cpu") -> torch.Tensor:
        return make_hidden(self.L_tot, self.d, self.seed + 1, device)

    def weight(self, device="cpu") -> torch.Tensor:
        return make_weight(self.V, self.d, self.seed + 2, device)

    def flops(self, M: int) -> int:
        return 2 * M * self.V * self.d


def _w(name, **kw) -> Workload:
    return Workload(name=name, **kw)


# The five batch shapes. Seeds: 1000 + shape number (+ 10 * sub-index for ratio sweeps).
TINY = _w("tiny_L256_d256_V1024_r0.5_f32", B=1, L=256, d=256, V=1024, out_dtype="f32",
          chunk_rows=0, mask_kind="flat", r_m=0.5, seed=1000)
LLADA = [_w(f"llada8b_L4096_r{r}", B=1, L=4096, d=4096, V=126464, out_dtype="bf16",
            chunk_rows=0, mask_kind="flat", r_m=r, seed=1001 + 10 * i)
         for i, r in enumerate((0.1, 0.5, 0.9))]
DECODE = _w("block_decode_16x2048_blk32", B=16, L=2048, d=4096, V=126464, out_dtype="bf16",
            chunk_rows=0, mask_kind="block", block=32, seed=1002)
LONG = [_w(f"long_L131072_r{r}_chunk4096", B=1, L=131072, d=4096, V=126464, out_dtype="bf16",
           chunk_rows=4096, mask_kind="flat", r_m=r, seed=1003 + 10 * i)
        for i, r in enumerate((0.05, 0.3, 0.7, 0.9))]
DREAM = _w("dream7b_ragged_8x32768_chunk8192", B=8, L=32768, d=3584, V=152064, out_dtype="bf16",
           chunk_rows=8192, mask_kind="ragged", seed=1004)

# One launch of the Dream-shaped batch's chunk size (8192 masked rows of d = 3584 against
# V = 152,064), on hidden states small enough (65,536 rows) that a metric capture of it holds
# about 4 GB on the device: a profiling case, not one of the five batch shapes.
DREAM_CHUNK = _w("dream7b_chunk_L65536_M8192", B=1, L=65536, d=3584, V=152064, out_dtype="bf16",
                 chunk_rows=0, mask_kind="flat", r_m=0.125, seed=1005)

ALL = [TINY] + LLADA + [DECODE] + LONG + [DREAM]
BY_NAME = {w.name: w for w in ALL}
