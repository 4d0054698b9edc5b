"""Seeded synthetic inputs (gradient slices, master weights, parameter shards).

This module holds no arithmetic of the ZeRO step: it only draws numbers.  The
same bytes feed the CUDA path and (copied to the host) the CPU oracle.

Every stream is keyed by (seed, step, rank, partition, kind, block): values are
drawn with PyTorch's seeded generator on the target device in fixed blocks of
BLOCK elements, each block from its own generator seed, so that any tensor can
be regenerated piecewise.  Draws are float32 N(0, 1) scaled by std (and by the
loss scale for fp16 gradients), then rounded to the storage dtype.
"""
import random
from typing import Iterable, List, Optional, Sequence, Tuple

import torch

BLOCK = 1 << 24
KINDS = {"grad": 1, "master": 2, "inject": 3, "shard": 4, "misc": 5}
LP_DTYPES = {0: torch.float16, 1: torch.bfloat16}
_M64 = (1 << 64) - 1


def _mix64(z: int) -> int:
    """SplitMix64 finaliser (Steele, Lea & Flood, 2014)."""
    z = (z + 0x9E3779B97F4A7C15) & _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def stream_seed(seed: int, *key: int) -> int:
    h = _mix64(seed & _M64)
    for k in key:
        h = _mix64(h ^ (int(k) & _M64))
    return h & ((1 << 63) - 1)


def normal_(out: torch.Tensor, std: float, seed: int, *key: int) -> torch.Tensor:
    """Fill the 1-D tensor `out` with std * N(0, 1) draws, block by block."""
    assert out.dim() == 1
    gen = torch.Generator(device=out.device)
    n = out.numel()
    for b, b0 in enumerate(range(0, n, BLOCK)):
        b1 = min(n, b0 + BLOCK)
        gen.manual_seed(stream_seed(seed, *key, b))
        tmp = torch.randn(b1 - b0, generator=gen, device=out.device, dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        out[b0:b1].copy_(tmp)
    return out


def zero_outside(out: torch.Tensor, keep: Sequence[Tuple[int, int]]) -> torch.Tensor:
    """Zero every element of the 1-D tensor `out` not covered by the sorted,
    disjoint (start, length) ranges in `keep` (padding is not a parameter)."""
    pos = 0
    for start, length in sorted(keep):
        if start > pos:
            out[pos:start].zero_()
        pos = max(pos, start + length)
    if pos < out.numel():
        out[pos:].zero_()
    return out


def grad_slice(length: int, lp: int, std: float, scale: float, seed: int, step: int,
               src_rank: int, partition: int, device, keep=None) -> torch.Tensor:
    """Rank `src_rank`'s gradient over partition `partition`'s region, as
    std * scale * N(0, 1) in fp16 (lp=0) or bf16 (lp=1)."""
    out = torch.empty(length, dtype=LP_DTYPES[lp], device=device)
    normal_(out, std * scale, seed, step, src_rank, partition, KINDS["grad"])
    if keep is not None:
        zero_outside(out, keep)
    return out


def master_init(length: int, std: float, seed: int, partition: int, device,
                keep=None) -> torch.Tensor:
    out = torch.empty(length, dtype=torch.float32, device=device)
    normal_(out, std, seed, 0, 0, partition, KINDS["master"])
    if keep is not None:
        zero_outside(out, keep)
    return out


def lp_shard(length: int, lp: int, std: float, seed: int, rank: int, device,
             keep=None) -> torch.Tensor:
    out = torch.empty(length, dtype=LP_DTYPES[lp], device=device)
    normal_(out, std, seed, 0, rank, 0, KINDS["shard"])
    if keep is not None:
        zero_outside(out, keep)
    return out


def inject_position(seed: int, step: int, partition: int, n_ranks: int,
                    keep: Iterable[Tuple[int, int]]) -> Tuple[int, int]:
    """A seeded (slice j, element i) inside the kept (non-padding) ranges."""
    rng = random.Random(stream_seed(seed, step, 0, partition, KINDS["inject"]))
    ranges: List[Tuple[int, int]] = [(s, n) for s, n in keep if n > 0]
    total = sum(n for _, n in ranges)
    k = rng.randrange(total)
    j = rng.randrange(n_ranks)
    for s, n in ranges:
        if k < n:
            return j, s + k
        k -= n
    raise AssertionError("unreachable")


def to_numpy_codes(t: torch.Tensor):
    """Raw 16-bit codes of an fp16/bf16 tensor as a host numpy uint16 array."""
    import numpy as np
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def to_numpy(t: torch.Tensor):
    return t.detach().cpu().numpy()


def pinned_like(t: torch.Tensor, pin: Optional[bool] = True) -> torch.Tensor:
    return torch.empty(t.shape, dtype=t.dtype, device="cpu", pin_memory=bool(pin))
