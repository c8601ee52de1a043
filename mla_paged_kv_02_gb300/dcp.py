"""Decode context parallelism (DCP): the latent cache of every request is split by
sequence across ranks.

Each rank holds a contiguous, page-aligned range of every request's tokens in
its own paged cache, attends over that range with all query rows of the batch
(``mla_decode_shard``), and the ranks' 513-wide (o, lse) partials are
all-gathered and merged by LSE (``mla_combine_shards``).  This is the
sequence-sharded decode the vLLM PR #46819 summary sizes its split partials
for (key code excerpt: ``q_num_heads = num_heads * dcp_world_size``) and the
vLLM PR #47327 report's DCP-aware workspace (implementation breakdown 1).

Everything here is host-side bookkeeping (which tokens a rank holds, its local
block table) plus the one exchange, an all-gather over ``torch.distributed``;
the attention and the merge run in the CUDA library.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import torch

from . import _lib

PAGE_SIZE = 64


def shard_bounds(seq_lens: Sequence[int], world: int, rank: int) -> List[Tuple[int, int]]:
    """[start, end) of every request's tokens that ``rank`` holds.

    Request b's ceil(L_b / 64) pages are cut into ``world`` contiguous runs of
    as equal a page count as possible (earlier ranks take the extra pages), so
    every range starts on a page boundary and a rank's pages are whole pages of
    the request.  A rank may hold nothing of a short request."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    out = []
    for L in seq_lens:
        L = int(L)
        pages = -(-L // PAGE_SIZE)
        base, extra = divmod(pages, world)
        p0 = rank * base + min(rank, extra)
        p1 = p0 + base + (1 if rank < extra else 0)
        out.append((min(p0 * PAGE_SIZE, L), min(p1 * PAGE_SIZE, L)))
    return out


def local_block_table(block_table: torch.Tensor, bounds: Sequence[Tuple[int, int]]) -> torch.Tensor:
    """The rank's block table: row b lists the pages of its tokens [start, end) of
    request b, so local token t lies at local page t // 64, slot t % 64 (ranges
    start on page boundaries).  Entries past a request's local pages are -1."""
    B = block_table.shape[0]
    n_local = [-(-(e - s) // PAGE_SIZE) for s, e in bounds]
    width = max(1, max(n_local) if n_local else 1)
    out = torch.full((B, width), -1, dtype=torch.int32, device=block_table.device)
    for b, ((s, _), n) in enumerate(zip(bounds, n_local)):
        if n:
            p0 = s // PAGE_SIZE
            out[b, :n] = block_table[b, p0:p0 + n]
    return out


def gather_partials(partial: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather every rank's [B, q, H, 513] partial into [world, B, q, H, 513]
    (shard-major).  With no process group the world is this rank alone."""
    import torch.distributed as dist

    if group is None and not (dist.is_available() and dist.is_initialized()):
        return partial.unsqueeze(0)
    world = dist.get_world_size(group)
    out = torch.empty((world,) + tuple(partial.shape), dtype=partial.dtype, device=partial.device)
    dist.all_gather(list(out.unbind(0)), partial.contiguous(), group=group)
    return out


def decode(pl: _lib.Plan, q_nope, q_pe, kv_cache, block_table, shard_lens, shard_start, seq_lens,
           softmax_scale: float, kv_scale, out, lse, workspace, group=None, stream=None,
           shard_partial: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One DCP decode step on this rank: its shard's partial, the all-gather, the merge.

    ``pl`` is planned with max_seq_len >= every shard_lens[b].  Returns the
    gathered partials [world, B, q, H, 513]; ``out`` / ``lse`` receive the merged
    result on every rank."""
    B, q, H = q_nope.shape[0], q_nope.shape[1], q_nope.shape[2]
    if shard_partial is None:
        shard_partial = torch.empty((B, q, H, 513), dtype=torch.float32, device=q_nope.device)
    st = _lib.decode_shard(pl, q_nope.reshape(-1, q_nope.shape[-1]), q_pe.reshape(-1, q_pe.shape[-1]),
                           kv_cache, block_table, shard_lens, shard_start, seq_lens, softmax_scale, kv_scale,
                           shard_partial, workspace, stream)
    if st != _lib.MLA_OK:
        raise _lib.MlaError(st, "mla_decode_shard")
    parts = gather_partials(shard_partial, group)
    st = _lib.combine_shards(parts, out, lse, stream)
    if st != _lib.MLA_OK:
        raise _lib.MlaError(st, "mla_combine_shards")
    return parts
