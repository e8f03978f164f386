"""pa_decode on the GPU against the fp64 oracle (max-abs <= 1e-2, mean-abs <= 1e-3)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_03_gb300 as pa
from paged_kv_attention_03_gb300.inputs import (SMALL_WORKLOADS, WORKLOADS, Workload,
                                                bf16_bits, make_case, make_case_from_lengths,
                                                split_mixed)

from _parity import (assert_parity, device_tensors, host_inputs, oracle_attention,
                     oracle_store, rows_of)

pytestmark = pytest.mark.gpu


def _decode_case(case, dev, seqs=None, num_splits=0, window=None, fused_store=True):
    """Run store + decode for the decode sequences `seqs` of `case` on the GPU."""
    w = case.workload
    win = w.sliding_window if window is None else window
    seqs = np.arange(case.num_seqs) if seqs is None else np.asarray(seqs)
    assert (case.query_lens[seqs] == 1).all()
    rows = torch.as_tensor(case.cu_seqlens_q[seqs], dtype=torch.long, device=dev)
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=dev)
    q = case.q[rows].contiguous()
    key, value = case.key[rows].contiguous(), case.value[rows].contiguous()
    slots = t(case.slot_mapping[case.cu_seqlens_q[seqs]])
    max_len = int(case.seq_lens[seqs].max()) if len(seqs) else 0
    if not fused_store:
        pa.pa_store_kvcache(key, value, case.k_cache, case.v_cache, slots)
        key = value = slots = None
    out = pa.pa_decode(q, case.k_cache, case.v_cache, t(case.block_table[seqs]),
                       t(case.seq_lens[seqs]), max_len, w.final_scale, win, num_splits,
                       key=key, value=value, slot_mapping=slots)
    return out


def _full_check(case, dev, num_splits=0, window=None):
    h = host_inputs(case)
    oracle_store(case, h)
    ref = oracle_attention(case, h, window=window)
    out = _decode_case(case, dev, num_splits=num_splits, window=window)
    assert pa.pa_read_device_error(device=dev) == 0
    np.testing.assert_array_equal(bf16_bits(case.k_cache), h["k_cache"])
    np.testing.assert_array_equal(bf16_bits(case.v_cache), h["v_cache"])
    return assert_parity(out, ref, f"{case.workload.name} splits={num_splits}")


@pytest.mark.parametrize("name", ["tiny_decode", "batched_decode_small", "long_decode_small"])
def test_decode_small_workloads(cuda, name):
    _full_check(make_case(name, seed=31, device=cuda), cuda)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64])
def test_decode_split_count_does_not_change_result(cuda, splits):
    _full_check(make_case("long_decode_small", seed=32, device=cuda), cuda, num_splits=splits)


def test_decode_tiny_workload_exact_config(cuda):
    # 4 sequences of {17, 33, 64, 100} keys, 8/2 heads, D=64, scale 1/8, 64-block pool.
    case = make_case("tiny_decode", seed=0, device=cuda)
    assert list(case.seq_lens) == [17, 33, 64, 100] and case.num_blocks == 64
    _full_check(case, cuda)


@pytest.mark.parametrize("window", [1, 15, 16, 17, 100, 5000])
def test_decode_sliding_window(cuda, window):
    _full_check(make_case("batched_decode_small", seed=33, device=cuda), cuda, window=window)


@pytest.mark.parametrize("bs", [1, 8, 32, 64, 256])
def test_decode_block_sizes(cuda, bs):
    w = Workload("bs", 8, 2, 128, bs, ())
    case = make_case_from_lengths(w, [0, 6, 15, 16, 31, 200, 511], [1] * 7, seed=34,
                                  device=cuda)
    _full_check(case, cuda)
    _full_check(make_case_from_lengths(w, [40, 300], [1, 1], seed=35, device=cuda), cuda,
                num_splits=3, window=77)


@pytest.mark.parametrize("H,Hkv,D", [(8, 8, 128), (40, 8, 128), (16, 1, 64), (20, 1, 128),
                                     (64, 2, 64), (6, 3, 64), (24, 2, 128), (36, 4, 64)])
def test_decode_group_sizes_and_head_dims(cuda, H, Hkv, D):
    w = Workload("g", H, Hkv, D, 16, ())
    case = make_case_from_lengths(w, [0, 1, 14, 15, 16, 17, 333], [1] * 7, seed=36, device=cuda)
    _full_check(case, cuda)
    _full_check(case, cuda, num_splits=4)


def test_decode_zero_length_sequence_gives_zeros(cuda):
    w = Workload("z", 8, 2, 128, 16, ())
    case = make_case_from_lengths(w, [10, 30], [1, 1], seed=37, device=cuda)
    t = lambda a: torch.as_tensor(a, dtype=torch.int32, device=cuda)
    for splits in (1, 3):
        out = pa.pa_decode(case.q, case.k_cache, case.v_cache, t(case.block_table),
                           t([0, 31]), 31, w.final_scale, 0, splits)
        h = host_inputs(case)
        ref = oracle.paged_attention(h["q"][1:2], h["k_cache"], h["v_cache"],
                                     np.array([0, 1], np.int32), np.array([31], np.int32),
                                     case.block_table[1:2], 8, 2, 0, w.final_scale)
        assert not out[0].float().abs().sum().item()
        assert_parity(out[1:2], ref)
    assert pa.pa_read_device_error(device=cuda) == 0


def test_decode_bad_block_index_is_flagged_not_faulted(cuda):
    w = Workload("bad", 8, 2, 128, 16, ())
    case = make_case_from_lengths(w, [40, 20], [1, 1], seed=38, device=cuda)
    bt = case.block_table.copy()
    bt[0, 1] = case.num_blocks + 100  # a visible page points past the pool
    t = lambda a: torch.as_tensor(a, dtype=torch.int32, device=cuda)
    out = pa.pa_decode(case.q, case.k_cache, case.v_cache, t(bt), t(case.seq_lens), 41,
                       w.final_scale, 0, 2)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error(device=cuda) & pa.DEVERR_BLOCK_RANGE
    h = host_inputs(case)
    ref = oracle.paged_attention(h["q"][1:2], h["k_cache"], h["v_cache"],
                                 np.array([0, 1], np.int32), case.seq_lens[1:2],
                                 case.block_table[1:2], 8, 2, 0, w.final_scale)
    assert_parity(out[1:2], ref)  # the other sequence is unaffected


def test_decode_seq_len_beyond_declared_max_is_flagged(cuda):
    w = Workload("cap", 8, 2, 128, 16, ())
    case = make_case_from_lengths(w, [40], [1], seed=39, device=cuda)
    t = lambda a: torch.as_tensor(a, dtype=torch.int32, device=cuda)
    pa.pa_decode(case.q, case.k_cache, case.v_cache, t(case.block_table), t(case.seq_lens), 20,
                 w.final_scale, 0, 1)
    assert pa.pa_read_device_error(device=cuda) & pa.DEVERR_SEQ_RANGE


def _whole_batch_check(case, dev, seqs, what):
    """Store + decode of the decode sequences `seqs` in one launch configuration (the
    benchmark's), every output row compared with the oracle."""
    h = host_inputs(case)
    rows = case.cu_seqlens_q[np.asarray(seqs)]  # the decode tokens only
    oracle.store_kvcache(np.ascontiguousarray(h["key"][rows]),
                         np.ascontiguousarray(h["value"][rows]), h["k_cache"], h["v_cache"],
                         np.ascontiguousarray(case.slot_mapping[rows]), case.workload.block_size)
    out = _decode_case(case, dev, seqs=seqs)
    assert pa.pa_read_device_error(device=dev) == 0
    np.testing.assert_array_equal(bf16_bits(case.k_cache), h["k_cache"])
    np.testing.assert_array_equal(bf16_bits(case.v_cache), h["v_cache"])
    ref = oracle_attention(case, h, seqs=np.asarray(seqs))
    return assert_parity(out, ref, f"full size {what}")


def test_decode_full_size_batched(cuda):
    # Batch 64, 32/8 heads, D=128, seq_len U[512, 4096], 32768-block pool: the launch
    # configuration the benchmark times; every sequence and head checked.
    case = make_case("batched_decode", seed=0, device=cuda)
    _whole_batch_check(case, cuda, np.arange(case.num_seqs), "batched_decode")


def test_decode_full_size_long_context(cuda):
    # Batch 8, 40/8 heads (group of 5), seq_len U[32768, 131072].
    case = make_case("long_decode", seed=0, device=cuda)
    _whole_batch_check(case, cuda, np.arange(case.num_seqs), "long_decode")


def test_decode_full_size_tiny(cuda):
    # 4 sequences of {17, 33, 64, 100} keys, 8/2 heads, D=64, scale 1/8.
    case = make_case("tiny_decode", seed=0, device=cuda)
    _whole_batch_check(case, cuda, np.arange(case.num_seqs), "tiny_decode")


def test_decode_full_size_mixed_batch_decode_half(cuda):
    # The 128 decodes of the mixed workload, sliding window 4096.
    case = make_case("mixed_window", seed=0, device=cuda)
    _, dec = split_mixed(case)
    _whole_batch_check(case, cuda, dec, "mixed_window decodes (pa_decode)")
