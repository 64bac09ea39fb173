"""Splitting one prefill over GPUs by kv head, one process per GPU.

KAP and OSK read only a (request, kv head) group's own queries, keys and values (CoSA Sec. 4.2-4.3:
every score, selection and visit is per query head, and query head h reads kv head h / g), so the
groups are independent: rank r takes the contiguous kv heads [kv0, kv1) of ``kv_head_range`` and
their g query heads each, as contiguous per-rank tensors, and calls the unchanged C ABI on them.
No data crosses ranks during the computation.  A caller that needs the whole O on every rank
gathers it over heads afterwards (``gather_heads``); that is the only collective, and it is optional.

Layouts are the library's: q and out [T, Hq, d], caches [pages, P, Hkv, d].
"""
from __future__ import annotations

from typing import List, Sequence, Tuple


def kv_head_range(rank: int, world: int, num_kv_heads: int) -> Tuple[int, int]:
    """The kv heads [kv0, kv1) of ``rank`` out of ``world``: contiguous, disjoint, covering every head,
    sizes differing by at most one (the first num_kv_heads % world ranks take one more)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of world {world}")
    if world > num_kv_heads:
        raise ValueError(f"{world} ranks for {num_kv_heads} kv heads: some rank would have no head")
    base, extra = divmod(num_kv_heads, world)
    kv0 = rank * base + min(rank, extra)
    return kv0, kv0 + base + (1 if rank < extra else 0)


def q_head_range(kv0: int, kv1: int, group: int) -> Tuple[int, int]:
    """Query heads served by kv heads [kv0, kv1) when each kv head serves ``group`` query heads."""
    return kv0 * group, kv1 * group


def _contig(x):
    return x.contiguous() if hasattr(x, "contiguous") else __import__("numpy").ascontiguousarray(x)


def shard_heads(q, k_cache, v_cache, kv0: int, kv1: int, group: int):
    """Contiguous copies of the query heads and kv heads of one rank (torch tensors or numpy arrays).
    Local query head i of the shard reads local kv head i // group, as in the whole problem."""
    h0, h1 = q_head_range(kv0, kv1, group)
    return (_contig(q[:, h0:h1, :]), _contig(k_cache[:, :, kv0:kv1, :]),
            None if v_cache is None else _contig(v_cache[:, :, kv0:kv1, :]))


def gather_heads(out_local, world: int, num_kv_heads: int, group: int, process_group=None):
    """O [T, Hq, d] of the whole problem from every rank's O [T, Hq_r, d] (torch.distributed
    all_gather; ranks with fewer heads are padded for the exchange and trimmed after)."""
    import torch
    import torch.distributed as dist
    sizes: List[int] = []
    for r in range(world):
        a, b = kv_head_range(r, world, num_kv_heads)
        sizes.append((b - a) * group)
    hmax = max(sizes)
    T, h, d = out_local.shape
    buf = out_local
    if h < hmax:
        buf = torch.zeros((T, hmax, d), dtype=out_local.dtype, device=out_local.device)
        buf[:, :h] = out_local
    parts = [torch.empty_like(buf) for _ in range(world)]
    dist.all_gather(parts, buf.contiguous(), group=process_group)
    return torch.cat([p[:, :n] for p, n in zip(parts, sizes)], dim=1)


def head_ranges(world: int, num_kv_heads: int) -> Sequence[Tuple[int, int]]:
    return [kv_head_range(r, world, num_kv_heads) for r in range(world)]
