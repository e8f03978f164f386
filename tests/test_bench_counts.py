"""The benchmark's work counts, pinned to the oracle's mask.

bench.py reports bytes and FLOPs of *algorithmic* work: the keys each query may see
(bottom-right causal plus the window, "transformers continuous_batching",
build_attention_mask; "vllm-npu 0.4.2 wheel diff", torch_sdpa.py,
_make_sliding_window_bias), K and V read once per kv head for decode, and 4·D FLOP per
visible (query, key) pair per head for prefill (a dot product and a weighted sum of
length D).  Its counter uses a closed form; here every count is the number of allowed
cells of the oracle's mask matrices, the mask the parity tests pin to the pages.
"""
import os
import sys

import numpy as np
import pytest

import oracle
from paged_kv_attention_03_gb300.inputs import Workload, make_case_from_lengths

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _mask_count(case, window):
    return sum(int(oracle.mask(int(sq), int(sk), window).sum())
               for sq, sk in zip(case.query_lens, case.seq_lens))


CASES = [
    # (heads, kv heads, head dim, window, context lengths, query lengths)
    (32, 8, 128, 0, [0, 5, 300, 1000], [200, 1, 129, 1]),   # prefill and decode rows
    (8, 2, 64, 0, [17, 33, 64, 100], [1, 1, 1, 1]),         # decode only
    (32, 8, 128, 100, [0, 250, 37], [300, 64, 1]),          # window shorter than the rows
    (40, 8, 128, 7, [3, 0], [1, 20]),                       # window of 7, G = 5
    (16, 4, 64, 1, [10, 0], [5, 9]),                        # window of 1: self only
]


@pytest.mark.parametrize("H,Hkv,D,window,ctx,ql", CASES)
def test_attended_keys_equal_the_oracle_mask(H, Hkv, D, window, ctx, ql):
    w = Workload("count", H, Hkv, D, 16, (), sliding_window=window)
    case = make_case_from_lengths(w, ctx, ql, seed=3, device="cpu")
    n = _mask_count(case, window)
    assert bench.attended_keys(case) == n
    assert bench.decode_kv_bytes(case) == n * Hkv * D * 2 * 2      # K and V, bf16
    assert bench.prefill_flops(case) == n * 4 * D * H              # QK^T and PV per head


def test_prefill_flops_count_every_multiply_add():
    # Tiny case, counted element by element: for each head, visible (row, key) pair and
    # dimension, one multiply-add of the dot product and one of the weighted sum.
    w = Workload("tiny", 4, 2, 8, 16, (), sliding_window=3)
    case = make_case_from_lengths(w, [2, 0], [3, 4], seed=4, device="cpu")
    flops = 0
    for sq, sk in zip(case.query_lens, case.seq_lens):
        m = oracle.mask(int(sq), int(sk), 3)
        for _h in range(w.num_heads):
            for r in range(m.shape[0]):
                for j in range(m.shape[1]):
                    if m[r, j]:
                        flops += 2 * w.head_dim + 2 * w.head_dim
    assert bench.prefill_flops(case) == flops


def test_cascade_physical_bytes_count_each_cache_row_once():
    # Requests sharing the first 4 blocks of their tables: the physical bytes are the
    # distinct cache rows their keys reach through the block table, counted once each.
    from paged_kv_attention_03_gb300.inputs import make_shared_prefix_case

    w = Workload("cas", 8, 2, 64, 16, ())
    prefix_blocks = 4
    case = make_shared_prefix_case(w, prefix_blocks, [5, 20, 1, 33], seed=6, device="cpu")
    rows = set()
    for b, L in enumerate(case.seq_lens):
        for j in range(int(L)):
            rows.add((int(case.block_table[b, j // w.block_size]), j % w.block_size))
    row_bytes = w.num_kv_heads * w.head_dim * 2 * 2
    logical, physical = bench.cascade_bytes(case, prefix_blocks * w.block_size)
    assert physical == len(rows) * row_bytes
    assert logical == int(case.seq_lens.sum()) * row_bytes
