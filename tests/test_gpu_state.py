"""pa_decode_state and pa_merge_states on the GPU against the fp64 oracle.

"05 Attention Backends", section 7.1 (split-KV partial results, merged) and section 8
(cascade: prefix and suffix attended apart, then combined).  The state rows carry the
same bar as the attention output (max-abs <= 1e-2, mean-abs <= 1e-3).  The log of the
softmax denominator is checked to 5e-3 absolute: the kernels sum bf16-rounded weights
(relative error <= 2^-9 each, so ln of the sum moves by at most ~2e-3) and use ex2.approx.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_03_gb300 as pa
from paged_kv_attention_03_gb300.inputs import Workload, bf16_bits, make_case_from_lengths

from _parity import assert_parity, host_inputs, oracle_attention

pytestmark = pytest.mark.gpu

LSE_ABS = 5e-3


def _t(a, dev):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=dev)


def _oracle_states(case, key_begin, window):
    w = case.workload
    q, kc, vc = bf16_bits(case.q), bf16_bits(case.k_cache), bf16_bits(case.v_cache)
    outs, lses = [], []
    for b in range(case.num_seqs):
        sk = int(case.seq_lens[b])
        if sk == 0:
            outs.append(np.zeros((w.num_heads, w.head_dim)))
            lses.append(np.full(w.num_heads, -np.inf))
            continue
        o, l = oracle.attend_row_state(q[case.cu_seqlens_q[b]], kc, vc, case.block_table[b],
                                       sk, sk - 1, int(key_begin[b]), w.num_heads,
                                       w.num_kv_heads, window, w.final_scale)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def _check_lse(got, ref):
    g = got.detach().cpu().double().numpy()
    empty = np.isneginf(ref)
    assert np.array_equal(np.isneginf(g), empty), "empty rows must have lse = -inf"
    if (~empty).any():
        assert np.abs(g[~empty] - ref[~empty]).max() <= LSE_ABS


def _decode_case(dev, H=32, Hkv=8, D=128, lens=(1, 17, 300, 1024, 2500), seed=80):
    w = Workload("st", H, Hkv, D, 16, ())
    return make_case_from_lengths(w, [n - 1 for n in lens], [1] * len(lens), seed=seed,
                                  device=dev)


@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("window", [0, 200])
def test_decode_state_matches_oracle(cuda, splits, window):
    case = _decode_case(cuda)
    L = case.seq_lens
    # key_begin: 0, inside, the last key, exactly L (empty) and past L (empty).
    kb = np.array([0, 5, 299, 1024, 9999], dtype=np.int32)
    st, lse = pa.pa_decode_state(case.q, case.k_cache, case.v_cache, _t(case.block_table, cuda),
                                 _t(L, cuda), int(L.max()), case.workload.final_scale, window,
                                 splits, key_begin=_t(kb, cuda))
    assert pa.pa_read_device_error(device=cuda) == 0
    ref_o, ref_l = _oracle_states(case, kb, window)
    assert_parity(st, ref_o, f"state splits={splits} window={window}")
    _check_lse(lse, ref_l)
    assert not st[3:].any()  # empty ranges give zero rows


def test_decode_state_without_key_begin_equals_decode(cuda):
    case = _decode_case(cuda, H=40, Hkv=8, seed=81)
    L, bt = _t(case.seq_lens, cuda), _t(case.block_table, cuda)
    st, lse = pa.pa_decode_state(case.q, case.k_cache, case.v_cache, bt, L,
                                 int(case.seq_lens.max()), case.workload.final_scale)
    out = pa.pa_decode(case.q, case.k_cache, case.v_cache, bt, L, int(case.seq_lens.max()),
                       case.workload.final_scale)
    # Same splits and arithmetic: the bf16 output is the state rounded.
    assert torch.equal(st.to(torch.bfloat16), out)


def test_merge_states_matches_oracle_merge(cuda):
    rng = np.random.default_rng(82)
    R, rows, D = 5, 300, 128
    states = rng.standard_normal((R, rows, D))
    lses = rng.standard_normal((R, rows)) * 20
    lses[1, ::3] = -np.inf   # some parts empty
    lses[:, 7] = -np.inf     # a row with no part at all
    st = torch.as_tensor(states, dtype=torch.float32, device=cuda)
    ls = torch.as_tensor(lses, dtype=torch.float32, device=cuda)
    out_state = torch.empty(rows, D, dtype=torch.float32, device=cuda)
    out_lse = torch.empty(rows, dtype=torch.float32, device=cuda)
    out = pa.pa_merge_states(st, ls, out_state=out_state, out_lse=out_lse)
    ref, ref_lse = oracle.merge_states(st.double().cpu().numpy(), ls.double().cpu().numpy())
    np.testing.assert_allclose(out_state.cpu().double().numpy(), ref, rtol=1e-5, atol=1e-5)
    fin = ~np.isneginf(ref_lse)
    np.testing.assert_allclose(out_lse.cpu().double().numpy()[fin], ref_lse[fin], rtol=0,
                               atol=1e-4)
    assert np.isneginf(out_lse.cpu().numpy()[7]) and not out_state[7].any()
    assert torch.equal(out, out_state.to(torch.bfloat16))


@pytest.mark.parametrize("D", [64, 128])
def test_two_states_merge_to_the_whole_attention(cuda, D):
    # Keys [0, c) as a sequence truncated at c, keys [c, L) through key_begin.
    case = _decode_case(cuda, H=16, Hkv=4, D=D, lens=(40, 333, 2048), seed=83)
    L = case.seq_lens
    cut = np.array([16, 100, 1999], dtype=np.int32)
    bt = _t(case.block_table, cuda)
    s1, l1 = pa.pa_decode_state(case.q, case.k_cache, case.v_cache, bt, _t(cut, cuda),
                                int(L.max()), case.workload.final_scale)
    s2, l2 = pa.pa_decode_state(case.q, case.k_cache, case.v_cache, bt, _t(L, cuda),
                                int(L.max()), case.workload.final_scale,
                                key_begin=_t(cut, cuda))
    out = pa.pa_merge_states(torch.stack([s1, s2]), torch.stack([l1, l2]))
    assert_parity(out, oracle_attention(case, host_inputs(case)), "merged halves")


@pytest.mark.parametrize("ranks", [2, 4])
def test_context_parallel_decode_emulated_on_one_gpu(cuda, ranks):
    # Each "rank" holds a slice of every sequence's context in its own paged cache with
    # its own block table and lengths; the query attends its local keys only, the local
    # states are gathered and merged.  Ranks run one after another (no kernel waits on
    # another), so one GPU stands in for all of them.
    w = Workload("dcp", 32, 8, 128, 16, ())
    lens = np.array([700, 4096, 33, 2001])
    case = make_case_from_lengths(w, list(lens - 1), [1] * len(lens), seed=84, device=cuda)
    bs = w.block_size
    states, lses = [], []
    for r in range(ranks):
        # Rank r owns the contiguous key range [L*r/R, L*(r+1)/R) of each sequence,
        # copied into a fresh local pool.
        starts = (lens * r) // ranks
        ends = (lens * (r + 1)) // ranks
        local_len = ends - starts
        nblk = (local_len + bs - 1) // bs
        pool_k = torch.zeros(int(nblk.sum()) + 1, bs, w.num_kv_heads, w.head_dim,
                             dtype=torch.bfloat16, device=cuda)
        pool_v = torch.zeros_like(pool_k)
        table = np.full((len(lens), max(1, int(nblk.max()))), -1, dtype=np.int32)
        nxt = 0
        for b in range(len(lens)):
            for j in range(int(local_len[b])):
                pos = int(starts[b]) + j
                src_blk = int(case.block_table[b, pos // bs])
                if j % bs == 0:
                    table[b, j // bs] = nxt
                    nxt += 1
                dst_blk = int(table[b, j // bs])
                pool_k[dst_blk, j % bs] = case.k_cache[src_blk, pos % bs]
                pool_v[dst_blk, j % bs] = case.v_cache[src_blk, pos % bs]
        s, l = pa.pa_decode_state(case.q, pool_k, pool_v, _t(table, cuda), _t(local_len, cuda),
                                  int(local_len.max()), w.final_scale)
        states.append(s)
        lses.append(l)
    assert pa.pa_read_device_error(device=cuda) == 0
    out = pa.pa_merge_states(torch.stack(states), torch.stack(lses))
    assert_parity(out, oracle_attention(case, host_inputs(case)), f"dcp x{ranks}")


def test_dcp_decode_single_rank_is_plain_decode(cuda):
    # Without a process group the context-parallel call is the local decode.
    from paged_kv_attention_03_gb300.dcp import dcp_decode

    case = _decode_case(cuda, seed=85)
    L, bt = _t(case.seq_lens, cuda), _t(case.block_table, cuda)
    out = dcp_decode(case.q, case.k_cache, case.v_cache, bt, L, int(case.seq_lens.max()),
                     case.workload.final_scale)
    assert_parity(out, oracle_attention(case, host_inputs(case)), "dcp x1")


@pytest.mark.parametrize("deal", ["contiguous", "interleave16", "interleave64"])
@pytest.mark.parametrize("window", [1, 100, 1500, 5000])
def test_context_parallel_decode_with_window(cuda, deal, window):
    # Ranks emulated on one GPU as above, each with its own local cache; the window is on
    # global positions, so each rank starts at its first visible local key.
    from paged_kv_attention_03_gb300.dcp import dcp_key_begin

    ranks = 3
    w = Workload("dcpw", 32, 8, 128, 16, ())
    lens = np.array([700, 4096, 33, 2001, 1])
    case = make_case_from_lengths(w, list(lens - 1), [1] * len(lens), seed=86, device=cuda)
    bs = w.block_size
    inter = 0 if deal == "contiguous" else int(deal[len("interleave"):])
    states, lses = [], []
    for r in range(ranks):
        if inter:
            owned = [np.nonzero((np.arange(L) // inter) % ranks == r)[0] for L in lens]
            starts = None
        else:
            st_, en_ = (lens * r) // ranks, (lens * (r + 1)) // ranks
            owned = [np.arange(a, b) for a, b in zip(st_, en_)]
            starts = torch.as_tensor(st_.astype(np.int32), device=cuda)
        local_len = np.array([len(o) for o in owned], dtype=np.int32)
        nblk = (local_len + bs - 1) // bs
        pool_k = torch.zeros(int(nblk.sum()) + 1, bs, w.num_kv_heads, w.head_dim,
                             dtype=torch.bfloat16, device=cuda)
        pool_v = torch.zeros_like(pool_k)
        table = np.full((len(lens), max(1, int(nblk.max()))), -1, dtype=np.int32)
        nxt = 0
        for b in range(len(lens)):
            for j, pos in enumerate(owned[b]):
                if j % bs == 0:
                    table[b, j // bs] = nxt
                    nxt += 1
                src_blk = int(case.block_table[b, pos // bs])
                pool_k[int(table[b, j // bs]), j % bs] = case.k_cache[src_blk, pos % bs]
                pool_v[int(table[b, j // bs]), j % bs] = case.v_cache[src_blk, pos % bs]
        kb = dcp_key_begin(_t(lens, cuda), window, r, ranks, inter, starts, _t(local_len, cuda))
        # the rule, written out: keys of this rank with global position < L - window
        want = [int(np.sum(o < max(0, L - window))) for o, L in zip(owned, lens)]
        assert kb.cpu().tolist() == want
        s, l = pa.pa_decode_state(case.q, pool_k, pool_v, _t(table, cuda), _t(local_len, cuda),
                                  max(1, int(local_len.max())), w.final_scale, key_begin=kb)
        states.append(s)
        lses.append(l)
    assert pa.pa_read_device_error(device=cuda) == 0
    out = pa.pa_merge_states(torch.stack(states), torch.stack(lses))
    assert_parity(out, oracle_attention(case, host_inputs(case), window=window),
                  f"dcp {deal} window {window}")
