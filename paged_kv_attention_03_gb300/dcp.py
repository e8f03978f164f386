"""Decode context parallelism across ranks.

"vLLM learning book, 05 Attention Backends", section 4 (the attention metadata carries
max_dcp_context_kv_len and dcp_context_kv_lens: for a long context, each rank of the
decode context-parallel group holds part of every sequence's cached keys).  Reading
taken: rank r keeps its share of sequence b's keys in its own paged cache (its own
block table and local length); the decode query attends those local keys, giving a
partial result per (sequence, head) -- a normalised row and ln of its softmax
denominator (pa_decode_state) -- and the ranks exchange these partial results and merge
them (pa_merge_states, section 7.1's split-KV merge).  The exchange is one all-gather of
[batch, heads, head_dim + 1] floats per rank.  For decode every cached key is visible
to the query, so how keys are dealt to ranks does not matter -- except under a sliding
window, which is defined on global positions: the query at global position L - 1 sees
keys L - w .. L - 1.  dcp_key_begin turns that bound into each rank's first visible local
key for the two deals it knows: contiguous ranges (rank r holds global positions
[start_r, start_r + local_len)), or chunks of `interleave` consecutive positions dealt
round-robin (position p on rank (p // interleave) % world); local keys keep the global
order in both.  The partial decode then runs from that key with no local window.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from ._lib import pa_decode_state, pa_merge_states


def _world(group) -> int:
    if not dist.is_available() or not dist.is_initialized():
        return 1
    return dist.get_world_size(group)


def gather_states(state: torch.Tensor, lse: torch.Tensor,
                  group=None) -> tuple[torch.Tensor, torch.Tensor]:
    """All-gather every rank's partial result: returns states [R, *state.shape] and
    lses [R, *lse.shape] in rank order (R = 1 without a process group)."""
    world = _world(group)
    if world == 1:
        return state.unsqueeze(0), lse.unsqueeze(0)
    # One message per rank: the rows and their lse side by side.
    packed = torch.cat([state.reshape(-1, state.shape[-1]),
                        lse.reshape(-1, 1).to(state.dtype)], dim=1).contiguous()
    parts = [torch.empty_like(packed) for _ in range(world)]
    dist.all_gather(parts, packed, group=group)
    allp = torch.stack(parts)
    states = allp[..., :-1].reshape((world,) + tuple(state.shape)).contiguous()
    lses = allp[..., -1].reshape((world,) + tuple(lse.shape)).contiguous().to(lse.dtype)
    return states, lses


def dcp_key_begin(global_seq_lens: torch.Tensor, sliding_window: int, rank: int, world: int,
                  interleave: int = 0, local_starts: torch.Tensor | None = None,
                  local_seq_lens: torch.Tensor | None = None) -> torch.Tensor:
    """This rank's first visible local key per sequence under a window of w keys: the
    number of its keys whose global position is below L - w (int32, on the lengths'
    device).  interleave > 0: chunks of that many positions dealt round-robin over the
    world; otherwise local_starts[b] is the global position of this rank's first key and
    local_seq_lens[b] the number of its keys."""
    lo = (global_seq_lens.to(torch.int64) - int(sliding_window)).clamp(min=0)
    if interleave > 0:
        cycle = int(interleave) * int(world)
        below = (lo // cycle) * interleave + (lo % cycle - rank * interleave).clamp(0, interleave)
    else:
        if local_starts is None or local_seq_lens is None:
            raise ValueError("dcp_key_begin: a contiguous deal needs local_starts and "
                             "local_seq_lens")
        below = torch.minimum((lo - local_starts.to(torch.int64)).clamp(min=0),
                              local_seq_lens.to(torch.int64))
    return below.to(torch.int32).contiguous()


def dcp_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
               block_table: torch.Tensor, local_seq_lens: torch.Tensor, max_local_len: int,
               scale: float, group=None, num_splits: int = 0,
               out: torch.Tensor | None = None, sliding_window: int = 0,
               global_seq_lens: torch.Tensor | None = None, interleave: int = 0,
               local_starts: torch.Tensor | None = None, rank: int | None = None,
               world: int | None = None) -> torch.Tensor:
    """Decode over keys spread across the ranks of `group`: this rank's cache holds
    local_seq_lens[b] keys of sequence b.  Every rank returns the full result [B, H, D].
    With sliding_window > 0, global_seq_lens and the deal (interleave, or local_starts)
    give each rank's first visible key (dcp_key_begin); rank / world default to the
    group's."""
    key_begin = None
    if sliding_window > 0:
        if global_seq_lens is None:
            raise ValueError("dcp_decode: a sliding window needs global_seq_lens")
        if rank is None:
            rank = dist.get_rank(group) if _world(group) > 1 else 0
        if world is None:
            world = _world(group)
        key_begin = dcp_key_begin(global_seq_lens, sliding_window, rank, world, interleave,
                                  local_starts, local_seq_lens)
    state, lse = pa_decode_state(q, k_cache, v_cache, block_table, local_seq_lens,
                                 max_local_len, scale, 0, num_splits, key_begin=key_begin)
    states, lses = gather_states(state, lse, group)
    return pa_merge_states(states, lses, out=out)
