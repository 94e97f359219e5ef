"""Multi-GPU partition of a layer: whole GQA groups per rank, no collective on the data path.

Every step of the path (estimation, index build, selection, attention) is independent per
q-head given its KV head, so a layer shards by whole GQA groups: rank r gets a contiguous
run of KV heads and the q-heads that read them, and its Q/K/V/O slices never leave it.  The
only cross-rank traffic is measurement: a barrier around the timed region and the maximum
of the ranks' times.
"""
from __future__ import annotations

from typing import List, Optional

__all__ = ["gqa_shard", "reduce_max", "layers_per_ms"]


def gqa_shard(Hq: int, Hkv: int, rank: int, world: int) -> List[int]:
    """The q-heads of rank ``rank``: whole GQA groups (consecutive KV heads), balanced so that
    group counts differ by at most one between ranks; ranks beyond Hkv get none."""
    if Hq <= 0 or Hkv <= 0 or Hq % Hkv:
        raise ValueError("Hq must be a positive multiple of Hkv")
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("rank must be in [0, world)")
    g = Hq // Hkv
    per, extra = divmod(Hkv, world)
    lo = rank * per + min(rank, extra)
    hi = lo + per + (1 if rank < extra else 0)
    return list(range(lo * g, hi * g))


def reduce_max(x: float, dist=None, device: Optional[str] = None) -> float:
    """Maximum of ``x`` over the ranks of the default process group (``x`` without one)."""
    if dist is None or not dist.is_initialized():
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def layers_per_ms(ms_max: float, world: int) -> float:
    """Whole-job time per layer when each of ``world`` ranks runs one layer replica per step
    and the slowest rank takes ``ms_max`` milliseconds."""
    return ms_max / world
