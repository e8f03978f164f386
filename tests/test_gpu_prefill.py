"""pa_varlen_prefill on the GPU against the fp64 oracle (max-abs <= 1e-2, mean-abs <= 1e-3)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_03_gb300 as pa
from paged_kv_attention_03_gb300.inputs import (SMALL_WORKLOADS, WORKLOADS, Workload,
                                                bf16_bits, make_case, make_case_from_lengths,
                                                split_mixed)

from _parity import (assert_parity, device_tensors, host_inputs, oracle_attention,
                     oracle_store)

pytestmark = pytest.mark.gpu


def _prefill(case, dev, window=None, fused_store=True, use_cu_k=False, both=False, out=None):
    w = case.workload
    win = w.sliding_window if window is None else window
    m = device_tensors(case, dev)
    key = value = slots = None
    if fused_store:
        key, value, slots = case.key, case.value, m["slot_mapping"]
    cu_k = None
    seq_lens = m["seq_lens"]
    if use_cu_k or both:
        cuk = np.zeros(case.num_seqs + 1, np.int32)
        cuk[1:] = np.cumsum(case.seq_lens)
        cu_k = torch.as_tensor(cuk, device=dev)
        if not both:
            seq_lens = None
    return pa.pa_varlen_prefill(case.q, case.k_cache, case.v_cache, m["cu_seqlens_q"], seq_lens,
                                m["block_table"], case.max_query_len, case.max_seq_len,
                                w.final_scale, win, cu_seqlens_k=cu_k, key=key, value=value,
                                slot_mapping=slots, out=out)


def _full_check(case, dev, window=None, what=None, **kw):
    h = host_inputs(case)
    oracle_store(case, h)
    ref = oracle_attention(case, h, window=window)
    out = _prefill(case, dev, window=window, **kw)
    flags = pa.pa_read_device_error(device=dev)
    assert flags == 0, f"device error bits {flags:#x}"
    np.testing.assert_array_equal(bf16_bits(case.k_cache), h["k_cache"])
    np.testing.assert_array_equal(bf16_bits(case.v_cache), h["v_cache"])
    return assert_parity(out, ref, what or case.workload.name)


@pytest.mark.parametrize("name", ["varlen_prefill_small", "mixed_window_small"])
def test_prefill_small_workloads(cuda, name):
    _full_check(make_case(name, seed=41, device=cuda), cuda)


def test_prefill_single_short_sequence(cuda):
    w = Workload("one", 8, 2, 128, 16, ())
    _full_check(make_case_from_lengths(w, [0], [1], seed=40, device=cuda), cuda)
    _full_check(make_case_from_lengths(w, [0], [40], seed=40, device=cuda), cuda)


@pytest.mark.parametrize("window", [0, 1, 7, 16, 100, 129, 300])
def test_prefill_windows_and_chunks(cuda, window):
    w = Workload("win", 32, 8, 128, 16, ())
    case = make_case_from_lengths(w, [0, 0, 37, 130, 500, 3], [1, 160, 64, 129, 31, 1], seed=42,
                                  device=cuda)
    _full_check(case, cuda, window=window)


@pytest.mark.parametrize("H,Hkv,D", [(8, 8, 128), (32, 8, 128), (40, 8, 128), (16, 2, 64),
                                     (64, 4, 128), (6, 3, 64), (128, 1, 64)])
def test_prefill_group_sizes_and_head_dims(cuda, H, Hkv, D):
    w = Workload("g", H, Hkv, D, 16, ())
    case = make_case_from_lengths(w, [0, 5, 100], [150, 17, 33], seed=43, device=cuda)
    _full_check(case, cuda)
    _full_check(case, cuda, window=50)


@pytest.mark.parametrize("bs", [16, 32, 64, 256])
def test_prefill_block_sizes(cuda, bs):
    w = Workload("bs", 16, 4, 128, bs, ())
    case = make_case_from_lengths(w, [0, 33, 250], [200, 15, 70], seed=44, device=cuda)
    _full_check(case, cuda)


@pytest.mark.parametrize("lens", [[16], [128], [127], [129], [255], [256], [257]])
def test_prefill_tile_edges(cuda, lens):
    w = Workload("edge", 32, 8, 128, 16, ())
    _full_check(make_case_from_lengths(w, [0] * len(lens), lens, seed=45, device=cuda), cuda)
    _full_check(make_case_from_lengths(w, [x // 2 for x in lens], [max(1, x // 3) for x in lens],
                                       seed=46, device=cuda), cuda)


@pytest.mark.parametrize("H,Hkv", [(8, 2), (32, 8)])
def test_prefill_many_sequences(cuda, H, Hkv):
    # 150 sequences of 1..300 query tokens (some with a cached context): the work list
    # has far more (query block, sequence) pairs than one 32-pair scan window, most of
    # the longest-first positions are empty, and every row is checked.
    w = Workload("many", H, Hkv, 128, 16, ())
    rng = np.random.default_rng(7)
    q = rng.integers(1, 301, size=150)
    ctx = np.where(rng.random(150) < 0.3, rng.integers(0, 200, size=150), 0)
    _full_check(make_case_from_lengths(w, ctx, q, seed=52, device=cuda), cuda)


def test_prefill_late_bad_sequence_is_flagged(cuda):
    # A sequence far down the work list with more queries than keys is reported too.
    w = Workload("late", 8, 2, 128, 16, ())
    case = make_case_from_lengths(w, [0] * 200, [40] * 200, seed=53, device=cuda)
    m = device_tensors(case, cuda)
    bad = case.seq_lens.copy()
    bad[187] = 10  # 40 queries, 10 keys
    pa.pa_read_device_error(clear=True, device=cuda)
    pa.pa_varlen_prefill(case.q, case.k_cache, case.v_cache, m["cu_seqlens_q"],
                         torch.as_tensor(bad, device=cuda), m["block_table"], 40, 40,
                         w.final_scale, 0)
    assert pa.pa_read_device_error(clear=True, device=cuda) & pa.DEVERR_QUERY_LEN


def test_prefill_cu_seqlens_k_instead_of_seq_lens(cuda):
    case = make_case("mixed_window_small", seed=47, device=cuda)
    _full_check(case, cuda, use_cu_k=True)


def test_prefill_cu_seqlens_k_disagreeing_is_flagged(cuda):
    case = make_case("varlen_prefill_small", seed=48, device=cuda)
    m = device_tensors(case, cuda)
    cuk = np.zeros(case.num_seqs + 1, np.int32)
    cuk[1:] = np.cumsum(case.seq_lens) + 1  # off by one
    w = case.workload
    pa.pa_varlen_prefill(case.q, case.k_cache, case.v_cache, m["cu_seqlens_q"], m["seq_lens"],
                         m["block_table"], case.max_query_len, case.max_seq_len, w.final_scale,
                         0, cu_seqlens_k=torch.as_tensor(cuk, device=cuda))
    assert pa.pa_read_device_error(device=cuda) & pa.DEVERR_SEQLENS_K


def test_prefill_bad_block_index_is_flagged_not_faulted(cuda):
    w = Workload("bad", 8, 2, 128, 16, ())
    case = make_case_from_lengths(w, [0, 0], [70, 40], seed=49, device=cuda)
    m = device_tensors(case, cuda)
    bt = case.block_table.copy()
    bt[0, 2] = case.num_blocks + 7
    pa.pa_varlen_prefill(case.q, case.k_cache, case.v_cache, m["cu_seqlens_q"], m["seq_lens"],
                         torch.as_tensor(bt, device=cuda), case.max_query_len, case.max_seq_len,
                         w.final_scale, 0)
    assert pa.pa_read_device_error(device=cuda) & pa.DEVERR_BLOCK_RANGE


def test_prefill_query_longer_than_keys_is_flagged(cuda):
    w = Workload("ql", 8, 2, 128, 16, ())
    case = make_case_from_lengths(w, [0, 10], [20, 5], seed=50, device=cuda)
    m = device_tensors(case, cuda)
    bad = torch.as_tensor(np.array([10, 15], np.int32), device=cuda)  # 20 queries, 10 keys
    pa.pa_varlen_prefill(case.q, case.k_cache, case.v_cache, m["cu_seqlens_q"], bad,
                         m["block_table"], 20, 20, w.final_scale, 0)
    assert pa.pa_read_device_error(device=cuda) & pa.DEVERR_QUERY_LEN


def test_prefill_stale_rows_past_the_sequence_are_ignored(cuda):
    # Poison every cache slot past each sequence's end with NaN: the result must not change.
    w = Workload("nan", 8, 2, 128, 16, ())
    case = make_case_from_lengths(w, [0, 20], [37, 3], seed=51, device=cuda)
    h = host_inputs(case)
    oracle_store(case, h)
    ref = oracle_attention(case, h)
    m = device_tensors(case, cuda)
    pa.pa_store_kvcache(case.key, case.value, case.k_cache, case.v_cache, m["slot_mapping"])
    for i in range(case.num_seqs):
        sk = int(case.seq_lens[i])
        last = int(case.block_table[i, (sk - 1) // 16])
        if sk % 16:
            case.k_cache[last, sk % 16:] = float("nan")
            case.v_cache[last, sk % 16:] = float("nan")
    out = pa.pa_varlen_prefill(case.q, case.k_cache, case.v_cache, m["cu_seqlens_q"],
                               m["seq_lens"], m["block_table"], case.max_query_len,
                               case.max_seq_len, w.final_scale, 0)
    assert_parity(out, ref)


def test_prefill_full_size_varlen(cuda):
    # 16 prompts of U[128, 2048] tokens, 32/8 heads, D=128, bs=16: the benchmark's launch
    # (store + prefill in one call); every output row checked.
    case = make_case("varlen_prefill", seed=0, device=cuda)
    _full_check(case, cuda, what="full size varlen_prefill")


def test_prefill_full_size_mixed_chunks(cuda):
    # 8 chunks of 512 over contexts U[1024, 8192] + 128 decodes, window 4096, in one call;
    # every output row (chunk rows and decode rows) checked.
    case = make_case("mixed_window", seed=0, device=cuda)
    _full_check(case, cuda, what="full size mixed_window (one pa_varlen_prefill call)")


def test_mixed_call_orders_later_stream_work_after_the_prefill(cuda):
    # Eight long prompts beside one decode row: the decode launch runs on the SMs the
    # prefill leaves free and finishes long before it, yet work queued on the stream after
    # the call (here a copy of the output) must see every prefill row.
    w = Workload("order", 32, 8, 128, 16, ())
    case = make_case_from_lengths(w, [0] * 8 + [300], [2048] * 8 + [1], seed=54, device=cuda)
    out = torch.full_like(case.q, float("nan"))
    _prefill(case, cuda, out=out)
    snap = out.clone()  # same stream, no synchronisation before it
    torch.cuda.synchronize()
    assert pa.pa_read_device_error(device=cuda) == 0
    assert not torch.isnan(out).any()
    assert torch.equal(snap.view(torch.int16), out.view(torch.int16))


def test_mixed_call_with_only_single_row_sequences(cuda):
    # Every sequence has one query row although max_seqlen_q says 4: the prefill kernel
    # has no item (one CTA, which exits) and the decode launch beside it does all rows.
    w = Workload("dec_only", 32, 8, 128, 16, ())
    case = make_case_from_lengths(w, [0, 15, 300, 2000], [1, 1, 1, 1], seed=55, device=cuda)
    h = host_inputs(case)
    oracle_store(case, h)
    ref = oracle_attention(case, h)
    m = device_tensors(case, cuda)
    out = pa.pa_varlen_prefill(case.q, case.k_cache, case.v_cache, m["cu_seqlens_q"],
                               m["seq_lens"], m["block_table"], 4, case.max_seq_len,
                               w.final_scale, 0, key=case.key, value=case.value,
                               slot_mapping=m["slot_mapping"])
    assert pa.pa_read_device_error(device=cuda) == 0
    assert_parity(out, ref, "single-row sequences, max_seqlen_q = 4")


def test_decode_only_batch_checks_its_lengths(cuda):
    # max_seqlen_q = 1: no prefill kernel runs, so the decode launch of the call checks
    # cu_seqlens_k against seq_lens itself.
    w = Workload("dec_chk", 8, 2, 128, 16, ())
    case = make_case_from_lengths(w, [10, 40, 7], [1, 1, 1], seed=56, device=cuda)
    m = device_tensors(case, cuda)
    cuk = np.zeros(case.num_seqs + 1, np.int32)
    cuk[1:] = np.cumsum(case.seq_lens)
    cuk[2:] += 1  # sequence 1 disagrees
    pa.pa_read_device_error(clear=True, device=cuda)
    out = pa.pa_varlen_prefill(case.q, case.k_cache, case.v_cache, m["cu_seqlens_q"],
                               m["seq_lens"], m["block_table"], 1, case.max_seq_len,
                               w.final_scale, 0, cu_seqlens_k=torch.as_tensor(cuk, device=cuda))
    assert pa.pa_read_device_error(clear=True, device=cuda) & pa.DEVERR_SEQLENS_K
    h = host_inputs(case)
    assert_parity(out, oracle_attention(case, h), "decode-only batch, cu_seqlens_k flagged")


@pytest.mark.parametrize("max_q", [1, 40])
def test_rows_beyond_q_are_flagged_not_touched(cuda, max_q):
    # cu_seqlens_q names rows past the end of q / out: those sequences are flagged and
    # skipped (no row outside q / out is read or written), the others are computed.
    w = Workload("rows", 8, 2, 128, 16, ())
    lens = [1, 1, 1] if max_q == 1 else [40, 40, 40]
    case = make_case_from_lengths(w, [20, 30, 50], lens, seed=57, device=cuda)
    m = device_tensors(case, cuda)
    rows = int(case.cu_seqlens_q[2])  # q and out hold only the first two sequences' rows
    q = case.q[:rows].contiguous()
    out = torch.full_like(q, float("nan"))
    pa.pa_read_device_error(clear=True, device=cuda)
    pa.pa_varlen_prefill(q, case.k_cache, case.v_cache, m["cu_seqlens_q"], m["seq_lens"],
                         m["block_table"], max_q, case.max_seq_len, w.final_scale, 0, out=out)
    assert pa.pa_read_device_error(clear=True, device=cuda) & pa.DEVERR_QUERY_LEN
    h = host_inputs(case)
    assert_parity(out, oracle_attention(case, h, seqs=[0, 1]), "rows within q")
