"""Seeded synthetic inputs for paged KV-cache attention.

This module only draws inputs: sequence lengths, shuffled block tables, the
slot_mapping of the new tokens, cu_seqlens and N(0, 1) bf16 values.  It holds none
of the attention arithmetic and imports neither the CUDA binding nor the oracle, so
both sides of a parity test are fed from here.

Conventions (one sequence = one request of a step):

* ``context_len`` tokens are already in the cache, ``query_len`` new tokens arrive
  this step, ``seq_len = context_len + query_len`` ("05 Attention Backends",
  section 4, the FlashAttentionMetadata diagram).  Decode is ``query_len == 1``.
* Each sequence owns ``ceil(seq_len / block_size)`` physical blocks taken in order
  from one seeded ``randperm`` of the pool, so tables are distinct and shuffled;
  unused table entries are ``-1``.
* The new token at absolute position ``p`` of sequence ``i`` goes to slot
  ``block_table[i, p // block_size] * block_size + p % block_size`` (the slot
  derivation of "05 Attention Backends", Q&A 2).
* Seeds: lengths and tables come from a CPU ``torch.Generator`` seeded with
  ``seed``; values from a generator seeded with ``seed + 1`` on the target device.
  The whole cache pool is filled with N(0, 1) values, so slots the new tokens will
  overwrite hold stale random data until the store runs.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    """Shape of one workload: a list of sequence groups over one cache pool."""

    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    # (count, context_len range inclusive, query_len) groups, in batch order.
    groups: tuple
    num_blocks: int | None = None  # None: exactly the blocks the sequences need
    sliding_window: int = 0  # <= 0: none
    fixed_context_lens: tuple | None = None  # overrides random lengths (tiny decode)
    scale: float | None = None  # None: 1/sqrt(head_dim)

    @property
    def final_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.head_dim)


# The five workloads of the task statement.  Lengths are "seq_len" for decode
# (context_len = seq_len - 1 tokens already cached, plus the new one) and, for the
# varlen prefill, the prompt length with nothing cached.
WORKLOADS = {
    # 4 sequences of {17, 33, 64, 100} keys, 8/2 heads, D=64, pool of 64 blocks.
    "tiny_decode": Workload("tiny_decode", 8, 2, 64, 16, ((4, None, 1),), num_blocks=64,
                            fixed_context_lens=(16, 32, 63, 99), scale=1.0 / 8.0),
    # Llama-3-8B-shaped layer: batch 64, seq_len ~ U[512, 4096], pool 32768 blocks.
    "batched_decode": Workload("batched_decode", 32, 8, 128, 16, ((64, (511, 4095), 1),),
                               num_blocks=32768),
    # 16 prompts of U[128, 2048] tokens, nothing cached, stored then attended.
    "varlen_prefill": Workload("varlen_prefill", 32, 8, 128, 16, ((16, (0, 0), (128, 2048)),)),
    # 8 chunks of 512 new tokens over contexts U[1024, 8192] plus 128 decodes over
    # contexts U[1024, 8192], sliding window 4096.
    "mixed_window": Workload("mixed_window", 32, 8, 128, 16,
                             ((8, (1024, 8192), 512), (128, (1024, 8192), 1)),
                             sliding_window=4096),
    # batch 8, seq_len ~ U[32768, 131072], 40/8 heads (5 query heads per kv head).
    "long_decode": Workload("long_decode", 40, 8, 128, 16, ((8, (32767, 131071), 1),)),
}

# Reduced variants: same structure and distributions, sizes the fp64 oracle finishes
# in seconds while still spanning several tiles and ragged tails.
SMALL_WORKLOADS = {
    "tiny_decode": WORKLOADS["tiny_decode"],
    "batched_decode_small": Workload("batched_decode_small", 32, 8, 128, 16,
                                     ((6, (100, 700), 1),), num_blocks=512),
    "varlen_prefill_small": Workload("varlen_prefill_small", 32, 8, 128, 16,
                                     ((4, (0, 0), (1, 300)),)),
    "mixed_window_small": Workload("mixed_window_small", 32, 8, 128, 16,
                                   ((2, (40, 400), 130), (5, (40, 400), 1)),
                                   sliding_window=160),
    "long_decode_small": Workload("long_decode_small", 40, 8, 128, 16,
                                  ((2, (3000, 6000), 1),)),
}


@dataclass
class PagedCase:
    """One synthetic step: new tokens, the cache they join and the attention metadata."""

    workload: Workload
    context_lens: np.ndarray  # [S] int32, tokens already cached
    query_lens: np.ndarray  # [S] int32, new tokens this step
    seq_lens: np.ndarray  # [S] int32 = context_lens + query_lens
    cu_seqlens_q: np.ndarray  # [S + 1] int32
    block_table: np.ndarray  # [S, max_blocks] int32, -1 padded
    slot_mapping: np.ndarray  # [Tq] int32
    num_blocks: int
    q: torch.Tensor  # [Tq, H, D] bf16
    key: torch.Tensor  # [Tq, Hkv, D] bf16 (new tokens)
    value: torch.Tensor  # [Tq, Hkv, D] bf16
    k_cache: torch.Tensor  # [NB, bs, Hkv, D] bf16, context tokens present
    v_cache: torch.Tensor
    extras: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.num_seqs else 0

    @property
    def max_query_len(self) -> int:
        return int(self.query_lens.max()) if self.num_seqs else 0


def _uniform_int(g: torch.Generator, lo: int, hi: int, n: int) -> np.ndarray:
    return torch.randint(lo, hi + 1, (n,), generator=g).numpy().astype(np.int64)


def make_case(workload: Workload | str, seed: int = 0, device: str | torch.device = "cpu",
              num_blocks: int | None = None) -> PagedCase:
    """Draw one step of ``workload`` (a Workload or a name in WORKLOADS/SMALL_WORKLOADS)."""
    if isinstance(workload, str):
        workload = WORKLOADS.get(workload) or SMALL_WORKLOADS[workload]
    w = workload
    g = torch.Generator().manual_seed(seed)
    ctx_parts, q_parts = [], []
    for count, ctx_range, qlen in w.groups:
        if w.fixed_context_lens is not None:
            ctx = np.asarray(w.fixed_context_lens, dtype=np.int64)
        else:
            ctx = _uniform_int(g, ctx_range[0], ctx_range[1], count)
        if isinstance(qlen, tuple):
            ql = _uniform_int(g, qlen[0], qlen[1], count)
        else:
            ql = np.full(count, qlen, dtype=np.int64)
        ctx_parts.append(ctx)
        q_parts.append(ql)
    context_lens = np.concatenate(ctx_parts)
    query_lens = np.concatenate(q_parts)
    return make_case_from_lengths(w, context_lens, query_lens, seed=seed, device=device,
                                  num_blocks=num_blocks, generator=g)


def make_case_from_lengths(w: Workload, context_lens, query_lens, seed: int = 0,
                           device: str | torch.device = "cpu", num_blocks: int | None = None,
                           generator: torch.Generator | None = None,
                           values: str = "normal") -> PagedCase:
    """Build a case from explicit per-sequence lengths (edge cases use this directly)."""
    g = generator if generator is not None else torch.Generator().manual_seed(seed)
    context_lens = np.asarray(context_lens, dtype=np.int64)
    query_lens = np.asarray(query_lens, dtype=np.int64)
    seq_lens = context_lens + query_lens
    bs = w.block_size
    blocks_per_seq = (seq_lens + bs - 1) // bs
    need = int(blocks_per_seq.sum())
    nb = num_blocks or w.num_blocks or max(need, 1)
    if need > nb:
        raise ValueError(f"{w.name}: sequences need {need} blocks, pool has {nb}")
    perm = torch.randperm(nb, generator=g).numpy().astype(np.int64)
    max_blocks = max(int(blocks_per_seq.max()) if len(seq_lens) else 0, 1)
    block_table = np.full((len(seq_lens), max_blocks), -1, dtype=np.int64)
    cursor = 0
    for i, nblk in enumerate(blocks_per_seq):
        block_table[i, :nblk] = perm[cursor:cursor + nblk]
        cursor += int(nblk)
    cu = np.zeros(len(seq_lens) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(query_lens)
    slots = np.empty(int(cu[-1]), dtype=np.int64)
    for i in range(len(seq_lens)):
        pos = np.arange(context_lens[i], seq_lens[i])
        slots[cu[i]:cu[i + 1]] = block_table[i, pos // bs] * bs + pos % bs

    dev = torch.device(device)
    gv = torch.Generator(device=dev).manual_seed(seed + 1)
    H, Hkv, D = w.num_heads, w.num_kv_heads, w.head_dim
    T = int(cu[-1])

    def draw(*shape):
        if values == "normal":
            return torch.randn(*shape, generator=gv, device=dev, dtype=torch.float32).to(
                torch.bfloat16)
        raise ValueError(values)

    q = draw(T, H, D)
    key = draw(T, Hkv, D)
    value = draw(T, Hkv, D)
    k_cache = torch.empty(nb, bs, Hkv, D, dtype=torch.bfloat16, device=dev)
    v_cache = torch.empty(nb, bs, Hkv, D, dtype=torch.bfloat16, device=dev)
    # Fill in slabs to bound the fp32 temporary on large pools.
    slab = max(1, (1 << 26) // (bs * Hkv * D))
    for c in (k_cache, v_cache):
        for s in range(0, nb, slab):
            e = min(nb, s + slab)
            c[s:e] = draw(e - s, bs, Hkv, D)
    i32 = lambda a: np.ascontiguousarray(a, dtype=np.int32)
    return PagedCase(w, i32(context_lens), i32(query_lens), i32(seq_lens), i32(cu),
                     i32(block_table), i32(slots), nb, q, key, value, k_cache, v_cache)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor (copied to host when needed)."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def make_shared_prefix_case(w: Workload, prefix_blocks: int, suffix_lens, seed: int = 0,
                            device: str | torch.device = "cpu") -> PagedCase:
    """Decode requests whose first `prefix_blocks` cache blocks are the same physical
    blocks (a cached prefix shared by every request, e.g. one system prompt), each with
    its own suffix of suffix_lens[b] keys; the query is the last token (seq_len =
    prefix + suffix).  The blocks each request first held for its prefix stay unused."""
    prefix = prefix_blocks * w.block_size
    lens = np.asarray(suffix_lens, dtype=np.int64) + prefix
    case = make_case_from_lengths(w, list(lens - 1), [1] * len(lens), seed=seed, device=device)
    case.block_table[1:, :prefix_blocks] = case.block_table[0, :prefix_blocks]
    return case


def split_mixed(case: PagedCase) -> tuple[np.ndarray, np.ndarray]:
    """Indices of the sequences with query_len > 1 and of the decode (query_len == 1) ones."""
    pre = np.nonzero(case.query_lens != 1)[0]
    dec = np.nonzero(case.query_lens == 1)[0]
    return pre, dec
