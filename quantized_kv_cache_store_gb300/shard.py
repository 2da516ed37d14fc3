"""One verify call split across the ranks of a process group (one GPU each).

Every (sequence, kv-head) is independent, and the split-KV decomposition of
"sycl-three-attempts-arc-b70" (section "Part 3: joint_matrix + split-KV")
merges partial attention over disjoint token ranges by their log-sum-exps.
Two ways to spread one call over ranks follow from that:

* kv-head sharding: rank r owns kv-heads ``head_range(Hk, world, r)`` (their
  cache pages and their query heads) and computes their outputs; no data is
  exchanged (``gather_heads`` only assembles the full output where a caller
  wants it on every rank).
* sequence sharding: rank r owns a contiguous range of every sequence's
  pages (``page_ranges``); it computes the split-KV partials of its range
  (stage 1), the partials of all ranks are all-gathered along the split
  axis, and every rank merges them by log-sum-exp (stage 2).  The draft
  tokens (the last n_spec positions) always fall in the last rank's range,
  which is therefore the only one that applies the causal rule; every
  earlier position is visible to every draft.

The per-rank compute is a ``Backend``: ``GpuBackend`` calls the library's
stage 1 and stage 2 through the C ABI on the rank's GPU.  Host logic only
here: which pages each rank owns, its local block table and lengths, and the
exchange.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

BLOCK = 16


def head_range(Hk: int, world: int, rank: int) -> tuple[int, int]:
    """kv-heads [lo, hi) of rank ``rank``: contiguous, sizes differing by at most one."""
    if not 0 <= rank < world:
        raise ValueError("rank outside the group")
    base, extra = divmod(Hk, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


@dataclass(frozen=True)
class SeqShard:
    """Rank ``rank``'s part of every sequence: pages [page_lo[b], page_hi[b])."""
    rank: int
    world: int
    page_lo: np.ndarray     # int64 [B]
    page_hi: np.ndarray     # int64 [B]
    local_lens: np.ndarray  # int32 [B]: tokens of the range (the last rank's includes the drafts)
    causal: bool            # only the last rank's range holds drafts

    def block_table(self, block_table: np.ndarray) -> np.ndarray:
        """The rank's block table: row b lists the blocks of its page range
        (-1 past the end), so that local position p is global position
        16 page_lo[b] + p."""
        B = block_table.shape[0]
        width = max(1, int((self.page_hi - self.page_lo).max(initial=0)))
        out = np.full((B, width), -1, np.int32)
        for b in range(B):
            n = int(self.page_hi[b] - self.page_lo[b])
            out[b, :n] = block_table[b, self.page_lo[b]:self.page_hi[b]]
        return out


def page_ranges(seq_lens, n_spec: int, world: int, rank: int) -> SeqShard:
    """Cut every sequence's pages into ``world`` contiguous ranges of nearly
    equal size, the last range starting no later than the page of the first
    draft (so that all n_spec drafts are in it)."""
    L = np.asarray(seq_lens, np.int64)
    if np.any(L < n_spec):
        raise ValueError("every sequence holds its n_spec drafts")
    pages = (L + BLOCK - 1) // BLOCK
    first_draft_page = (L - n_spec) // BLOCK
    lo = np.empty_like(L)
    hi = np.empty_like(L)
    for b in range(L.shape[0]):
        # boundaries k * pages / world, the last one pulled back to the draft page
        cuts = [(pages[b] * k) // world for k in range(world + 1)]
        cuts[world - 1] = min(cuts[world - 1], first_draft_page[b])
        for k in range(world - 2, 0, -1):
            cuts[k] = min(cuts[k], cuts[k + 1])
        lo[b], hi[b] = cuts[rank], cuts[rank + 1]
    local = np.clip(np.minimum(L, hi * BLOCK) - lo * BLOCK, 0, None).astype(np.int32)
    return SeqShard(rank, world, lo, hi, local, causal=rank == world - 1)


class Backend:
    """The per-rank compute: stage 1 over the rank's range and the merge."""

    def stage1(self, q, block_table, seq_lens, num_kv_splits: int, causal: bool):
        """(partial_o [n_spec, B, Hq, S, 128], partial_lse [n_spec, B, Hq, S]) as tensors."""
        raise NotImplementedError

    def stage2(self, partial_o, partial_lse):
        """out [n_spec, B, Hq, 128]."""
        raise NotImplementedError


class GpuBackend(Backend):
    """tq_verify_stage1 / tq_verify_stage2 on the rank's GPU."""

    def __init__(self, cache: torch.Tensor, preset: int):
        self.cache = cache
        self.preset = preset

    def stage1(self, q, block_table, seq_lens, num_kv_splits, causal):
        from . import tqkv

        n, B, Hq, D = q.shape
        dev = self.cache.device
        po = torch.empty((n, B, Hq, num_kv_splits, D), dtype=torch.float32, device=dev)
        pl = torch.empty((n, B, Hq, num_kv_splits), dtype=torch.float32, device=dev)
        tqkv.tq_verify_stage1(self.cache, self.preset, q, torch.as_tensor(block_table, device=dev),
                              torch.as_tensor(seq_lens, dtype=torch.int32, device=dev), num_kv_splits, causal,
                              po, pl)
        return po, pl

    def stage2(self, partial_o, partial_lse):
        from . import tqkv

        n, B, Hq, _, D = partial_o.shape
        out = torch.empty((n, B, Hq, D), dtype=torch.float32, device=partial_o.device)
        tqkv.tq_verify_stage2(partial_o.contiguous(), partial_lse.contiguous(), out)
        return out


def verify_seq_sharded(backend: Backend, shard: SeqShard, q, block_table: np.ndarray,
                       num_kv_splits: int, group=None):
    """One verify call with the sequences' pages spread over the ranks of
    ``group`` (torch.distributed): stage 1 over this rank's range, an
    all-gather of the partials along the split axis (rank order = position
    order), and the log-sum-exp merge.  Every rank returns the full output."""
    import torch.distributed as dist

    po, pl = backend.stage1(q, shard.block_table(block_table), shard.local_lens, num_kv_splits, shard.causal)
    world = dist.get_world_size(group)
    pos = [torch.empty_like(po) for _ in range(world)]
    pls = [torch.empty_like(pl) for _ in range(world)]
    dist.all_gather(pos, po.contiguous(), group=group)
    dist.all_gather(pls, pl.contiguous(), group=group)
    return backend.stage2(torch.cat(pos, dim=3), torch.cat(pls, dim=3))


def gather_heads(out_local: torch.Tensor, Hk: int, group_size: int, group=None) -> torch.Tensor:
    """Assemble [n_spec, B, Hq, 128] on every rank from each rank's query heads
    (those of its kv-heads, ``head_range``)."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    n, B, _, D = out_local.shape
    sizes = [(head_range(Hk, world, r)[1] - head_range(Hk, world, r)[0]) * group_size for r in range(world)]
    width = max(sizes)
    pad = torch.zeros((n, B, width, D), dtype=out_local.dtype, device=out_local.device)
    pad[:, :, :out_local.shape[2]] = out_local
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad, group=group)
    return torch.cat([p[:, :, :s] for p, s in zip(parts, sizes)], dim=2)
