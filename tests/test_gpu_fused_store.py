"""Attention calls that also store the new tokens (key / value / slot_mapping given).

"05 Attention Backends", section 5: the attention call receives the new key and value
tensors with slot_mapping and writes the cache itself.  pa_decode does it inside its own
launch; pa_varlen_prefill stores first on the same stream.  Either way the result must
equal pa_store_kvcache followed by the attention without them: the same output bits and
the same cache bits.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_03_gb300 as pa
from paged_kv_attention_03_gb300.inputs import Workload, bf16_bits, make_case_from_lengths

from _parity import assert_parity, device_tensors, host_inputs, oracle_attention, oracle_store

pytestmark = pytest.mark.gpu


def _prefill(case, m, fused, window=0):
    w = case.workload
    kw = dict(key=case.key, value=case.value, slot_mapping=m["slot_mapping"]) if fused else {}
    if not fused:
        pa.pa_store_kvcache(case.key, case.value, case.k_cache, case.v_cache, m["slot_mapping"])
    return pa.pa_varlen_prefill(case.q, case.k_cache, case.v_cache, m["cu_seqlens_q"],
                                m["seq_lens"], m["block_table"], case.max_query_len,
                                case.max_seq_len, w.final_scale, window, **kw)


def _twin(case):
    """A second case object sharing the inputs but with its own copy of the caches."""
    import copy
    twin = copy.copy(case)
    twin.k_cache = case.k_cache.clone()
    twin.v_cache = case.v_cache.clone()
    return twin


# Contexts chosen so that the boundary between cached and new keys falls inside a
# 16-key piece (5, 300), on a piece boundary (32, 256), inside the first tile (0), and
# so that whole 128-key tiles are new (long queries); query length 1 is a decode row.
PREFILL_SHAPES = [
    ([0, 5, 32, 300], [200, 37, 1, 129]),
    ([256, 17, 1000], [1, 300, 64]),
]


@pytest.mark.parametrize("ctx,ql", PREFILL_SHAPES)
@pytest.mark.parametrize("window", [0, 100])
def test_prefill_fused_store_equals_separate_store(cuda, ctx, ql, window):
    w = Workload("f", 32, 8, 128, 16, ())
    case = make_case_from_lengths(w, ctx, ql, seed=71, device=cuda)
    other = _twin(case)
    m = device_tensors(case, cuda)
    fused = _prefill(case, m, True, window)
    assert pa.pa_read_device_error(device=cuda) == 0
    sep = _prefill(other, m, False, window)
    assert pa.pa_read_device_error(device=cuda) == 0
    assert torch.equal(fused, sep)
    assert torch.equal(case.k_cache, other.k_cache)
    assert torch.equal(case.v_cache, other.v_cache)
    h = host_inputs(other)
    ref = oracle_attention(case, h, window=window)
    assert_parity(fused, ref)


@pytest.mark.parametrize("H,Hkv,D", [(8, 8, 64), (40, 8, 128)])
def test_prefill_fused_store_head_shapes(cuda, H, Hkv, D):
    w = Workload("fh", H, Hkv, D, 16, ())
    case = make_case_from_lengths(w, [9, 0, 130], [70, 33, 5], seed=72, device=cuda)
    h = host_inputs(case)
    oracle_store(case, h)
    m = device_tensors(case, cuda)
    out = _prefill(case, m, True)
    assert pa.pa_read_device_error(device=cuda) == 0
    np.testing.assert_array_equal(bf16_bits(case.k_cache), h["k_cache"])
    np.testing.assert_array_equal(bf16_bits(case.v_cache), h["v_cache"])
    assert_parity(out, oracle_attention(case, h))


def test_prefill_with_store_overwrites_stale_new_rows(cuda):
    # Poison the cache rows of every new token with NaN: the call stores the new keys
    # before attending, so neither the result nor the final cache sees the poison.
    w = Workload("fn", 8, 2, 128, 16, ())
    case = make_case_from_lengths(w, [21, 0], [50, 140], seed=73, device=cuda)
    h = host_inputs(case)
    oracle_store(case, h)
    ref = oracle_attention(case, h)
    for t, slot in enumerate(case.slot_mapping):
        blk, off = divmod(int(slot), 16)
        case.k_cache[blk, off] = float("nan")
        case.v_cache[blk, off] = float("nan")
    m = device_tensors(case, cuda)
    out = _prefill(case, m, True)
    assert pa.pa_read_device_error(device=cuda) == 0
    assert_parity(out, ref)
    np.testing.assert_array_equal(bf16_bits(case.k_cache), h["k_cache"])
    np.testing.assert_array_equal(bf16_bits(case.v_cache), h["v_cache"])


@pytest.mark.parametrize("H,Hkv,D", [(8, 8, 64), (16, 16, 128)])
def test_prefill_fused_store_group_one_spans_three_tiles(cuda, H, Hkv, D):
    # G = 1: a work item is 256 query tokens, whose new keys reach over three 128-key tiles
    # (with a context of 7 the first and last only partly).
    w = Workload("g1", H, Hkv, D, 16, ())
    case = make_case_from_lengths(w, [7, 200, 0], [300, 257, 129], seed=80, device=cuda)
    other = _twin(case)
    m = device_tensors(case, cuda)
    fused = _prefill(case, m, True)
    assert pa.pa_read_device_error(device=cuda) == 0
    sep = _prefill(other, m, False)
    assert torch.equal(fused, sep)
    assert torch.equal(case.k_cache, other.k_cache)
    assert torch.equal(case.v_cache, other.v_cache)
    assert_parity(fused, oracle_attention(case, host_inputs(other)))


def test_prefill_fused_store_writes_rows_no_sequence_owns(cuda):
    # Rows of key / value before cu_seqlens_q[0] and from cu_seqlens_q[num_seqs] on belong
    # to no sequence: the store still writes those with a slot (and skips slot -1).
    w = Workload("fo", 8, 2, 128, 16, ())
    nb = 64
    case = make_case_from_lengths(w, [5, 40], [30, 70], seed=79, device=cuda, num_blocks=nb)
    used = set(case.block_table[case.block_table >= 0].ravel().tolist())
    free = [b for b in range(nb) if b not in used]
    front = [free[0] * 16 + 1, -1, free[0] * 16 + 7]
    back = [free[1] * 16, free[1] * 16 + 15, -1, free[2] * 16 + 3]
    g = torch.Generator(device=cuda).manual_seed(5)
    rnd = lambda n, heads: torch.randn(n, heads, 128, generator=g, device=cuda).to(torch.bfloat16)
    q = torch.cat([rnd(3, 8), case.q, rnd(4, 8)])
    key = torch.cat([rnd(3, 2), case.key, rnd(4, 2)])
    value = torch.cat([rnd(3, 2), case.value, rnd(4, 2)])
    slots = np.concatenate([front, case.slot_mapping, back]).astype(np.int32)
    h = host_inputs(case)
    oracle.store_kvcache(bf16_bits(key), bf16_bits(value), h["k_cache"], h["v_cache"], slots, 16)
    ref = oracle_attention(case, h)
    m = device_tensors(case, cuda)
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=cuda)
    out = pa.pa_varlen_prefill(q, case.k_cache, case.v_cache, t(case.cu_seqlens_q + 3),
                               m["seq_lens"], m["block_table"], case.max_query_len,
                               case.max_seq_len, w.final_scale, 0, key=key, value=value,
                               slot_mapping=t(slots))
    assert pa.pa_read_device_error(device=cuda) == 0
    np.testing.assert_array_equal(bf16_bits(case.k_cache), h["k_cache"])
    np.testing.assert_array_equal(bf16_bits(case.v_cache), h["v_cache"])
    assert_parity(out[3:3 + int(case.cu_seqlens_q[-1])], ref)
    # No sequence at all: nothing is attended, the rows are still stored.
    key2, value2 = rnd(2, 2), rnd(2, 2)
    slots2 = np.array([free[3] * 16 + 2, free[3] * 16 + 9], np.int32)
    oracle.store_kvcache(bf16_bits(key2), bf16_bits(value2), h["k_cache"], h["v_cache"], slots2, 16)
    pa.pa_varlen_prefill(rnd(2, 8), case.k_cache, case.v_cache, t([0]), t([]),
                         torch.zeros((0, 1), dtype=torch.int32, device=cuda), 0, 0,
                         w.final_scale, 0, key=key2, value=value2, slot_mapping=t(slots2))
    assert pa.pa_read_device_error(device=cuda) == 0
    np.testing.assert_array_equal(bf16_bits(case.k_cache), h["k_cache"])
    np.testing.assert_array_equal(bf16_bits(case.v_cache), h["v_cache"])


def _decode(case, dev, fused, splits=0, window=0):
    w = case.workload
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=dev)
    slots = t(case.slot_mapping)
    if not fused:
        pa.pa_store_kvcache(case.key, case.value, case.k_cache, case.v_cache, slots)
    kw = dict(key=case.key, value=case.value, slot_mapping=slots) if fused else {}
    return pa.pa_decode(case.q, case.k_cache, case.v_cache, t(case.block_table),
                        t(case.seq_lens), int(case.seq_lens.max()), w.final_scale, window,
                        splits, **kw)


@pytest.mark.parametrize("H,Hkv", [(32, 8), (64, 2)])  # G = 4; G = 32 (two head tiles)
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_decode_fused_store_equals_separate_store(cuda, H, Hkv, splits):
    w = Workload("fd", H, Hkv, 128, 16, ())
    case = make_case_from_lengths(w, [0, 15, 16, 700, 2047], [1, 1, 1, 1, 1], seed=75,
                                  device=cuda)
    other = _twin(case)
    fused = _decode(case, cuda, True, splits)
    assert pa.pa_read_device_error(device=cuda) == 0
    sep = _decode(other, cuda, False, splits)
    assert torch.equal(fused, sep)
    assert torch.equal(case.k_cache, other.k_cache)
    assert torch.equal(case.v_cache, other.v_cache)
    h = host_inputs(other)
    assert_parity(fused, oracle_attention(case, h))


def test_decode_fused_store_with_window(cuda):
    w = Workload("fw", 32, 8, 64, 16, ())
    case = make_case_from_lengths(w, [40, 900, 3], [1, 1, 1], seed=76, device=cuda)
    other = _twin(case)
    fused = _decode(case, cuda, True, 0, window=64)
    sep = _decode(other, cuda, False, 0, window=64)
    assert pa.pa_read_device_error(device=cuda) == 0
    assert torch.equal(fused, sep)
    assert torch.equal(case.k_cache, other.k_cache)


def test_decode_fused_slot_mismatch_is_flagged_and_empty_sequence_still_stored(cuda):
    w = Workload("fe", 8, 2, 128, 16, ())
    case = make_case_from_lengths(w, [10, 30], [1, 1], seed=77, device=cuda)
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=cuda)
    slots = t(case.slot_mapping[::-1])  # each token aimed at the other sequence's row
    pa.pa_decode(case.q, case.k_cache, case.v_cache, t(case.block_table), t(case.seq_lens),
                 int(case.seq_lens.max()), w.final_scale, 0, 0, key=case.key,
                 value=case.value, slot_mapping=slots)
    assert pa.pa_read_device_error(device=cuda) & pa.DEVERR_SLOT_MISMATCH
    # A sequence with no keys: nothing reads its new row, which is still written.
    case2 = make_case_from_lengths(w, [10, 30], [1, 1], seed=78, device=cuda)
    slot = int(case2.slot_mapping[0])
    pa.pa_decode(case2.q, case2.k_cache, case2.v_cache, t(case2.block_table), t([0, 31]), 31,
                 w.final_scale, 0, 0, key=case2.key, value=case2.value,
                 slot_mapping=t(case2.slot_mapping))
    pa.pa_read_device_error(device=cuda)  # a zero-length sequence with a slot is flagged
    blk, off = divmod(slot, 16)
    assert torch.equal(case2.k_cache[blk, off], case2.key[0])
    assert torch.equal(case2.v_cache[blk, off], case2.value[0])
