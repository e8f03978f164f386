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
to the query, so how keys are dealt to ranks does not matter; a sliding window (defined
on global positions) is not supported here.
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


def dcp_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
               block_table: torch.Tensor, local_seq_lens: torch.Tensor, max_local_len: int,
               scale: float, group=None, num_splits: int = 0,
               out: torch.Tensor | None = None) -> torch.Tensor:
    """Decode over keys spread across the ranks of `group`: this rank's cache holds
    local_seq_lens[b] keys of sequence b.  Every rank returns the full result [B, H, D]."""
    state, lse = pa_decode_state(q, k_cache, v_cache, block_table, local_seq_lens,
                                 max_local_len, scale, 0, num_splits)
    states, lses = gather_states(state, lse, group)
    return pa_merge_states(states, lses, out=out)
