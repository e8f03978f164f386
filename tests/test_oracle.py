"""Pins of the fp64 CPU oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: each test checks it against a worked
example printed on a page (tests/golden/), a different formulation printed on a
page (the HF diagonal formulas, the torch_sdpa tril/triu window), a library routine
(torch scaled_dot_product_attention in fp64), a closed form, or an invariant that a
plausible slip (dropped scale, wrong GQA mapping, wrong block/offset split, top-left
instead of bottom-right causal alignment, off-by-one window) would break.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_03_gb300.inputs import (SMALL_WORKLOADS, Workload, bf16_bits,
                                                make_case, make_case_from_lengths)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden_mask(name):
    rows, header = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if header is None:
                header = dict(kv.split("=") for kv in line.split())
                continue
            rows.append([c == "1" for c in line])
    return int(header["sk"]), int(header["sq"]), int(header["window"]), np.array(rows)


# ------------------------------------------------------------------ masks ---

@pytest.mark.parametrize("name", ["hf_mask_example_1.txt", "hf_mask_example_2.txt"])
def test_mask_matches_printed_examples(name):
    sk, sq, w, expect = _read_golden_mask(name)
    got = oracle.mask(sq, sk, w)
    assert got.shape == expect.shape
    np.testing.assert_array_equal(got, expect)


def _hf_formula_allowed(sq, sk, w):
    """build_attention_mask's diagonals ("transformers ... input_ouputs.py"), as printed:
    causal diagonal sk - sq + 1 when 1 <= sq < sk (else 1), triu of -inf above it; if
    w > 1 also tril of -inf at diagonal sk - sq - w."""
    causal_diagonal = sk - sq + 1 if 1 <= sq < sk else 1
    ones = torch.ones(sq, sk, dtype=torch.bool)
    masked = torch.triu(ones, diagonal=causal_diagonal)
    if w > 1:
        masked |= torch.tril(ones, diagonal=sk - sq - w)
    return (~masked).numpy()


@pytest.mark.parametrize("w", [0, 2, 3, 5, 8, 100])
def test_mask_matches_hf_diagonal_formulas(w):
    for sk in range(1, 14):
        for sq in range(1, sk + 1):
            np.testing.assert_array_equal(oracle.mask(sq, sk, w), _hf_formula_allowed(sq, sk, w),
                                          err_msg=f"sq={sq} sk={sk} w={w}")


@pytest.mark.parametrize("w", [1, 2, 4, 7, 20])
def test_square_window_matches_sdpa_bias(w):
    # torch_sdpa.py _make_sliding_window_bias: tril(ones, 0) then triu(., -w + 1).
    for n in range(1, 12):
        keep = torch.triu(torch.tril(torch.ones(n, n), diagonal=0), diagonal=-w + 1) > 0
        np.testing.assert_array_equal(oracle.mask(n, n, w), keep.numpy())


def test_window_one_is_self_only_and_rejects_more_queries_than_keys():
    np.testing.assert_array_equal(oracle.mask(3, 6, 1),
                                  np.array([[0, 0, 0, 1, 0, 0], [0, 0, 0, 0, 1, 0],
                                            [0, 0, 0, 0, 0, 1]], dtype=bool))
    with pytest.raises(oracle.OracleError):
        oracle.mask(4, 3, 0)


# ------------------------------------------------------------------ store ---

def test_store_matches_printed_example():
    with open(os.path.join(GOLDEN, "store_kvcache_example.txt")) as f:
        lines = [l.strip() for l in f if l.strip() and not l.startswith("#")]
    hdr = dict(kv.split("=") for kv in lines[0].split())
    T, hkv, d = int(hdr["num_tokens"]), int(hdr["num_kv_heads"]), int(hdr["head_dim"])
    nb, bs = int(hdr["num_blocks"]), int(hdr["block_size"])
    slots = np.array([int(x) for x in lines[1].split("=")[1].split(",")], dtype=np.int32)
    where = {int(a): int(b) for a, b in (l.split() for l in lines[2:])}
    g = torch.Generator().manual_seed(7)
    key = bf16_bits(torch.randn(T, hkv, d, generator=g).to(torch.bfloat16))
    value = bf16_bits(torch.randn(T, hkv, d, generator=g).to(torch.bfloat16))
    kc = np.zeros((nb, bs, hkv, d), np.uint16)
    vc = np.zeros((nb, bs, hkv, d), np.uint16)
    oracle.store_kvcache(key, value, kc, vc, slots, bs)
    flat_k, flat_v = kc.reshape(nb * bs, hkv, d), vc.reshape(nb * bs, hkv, d)
    written = set()
    for t, s in where.items():
        if s < 0:
            continue
        np.testing.assert_array_equal(flat_k[s], key[t])
        np.testing.assert_array_equal(flat_v[s], value[t])
        written.add(s)
    untouched = [s for s in range(nb * bs) if s not in written]
    assert not flat_k[untouched].any() and not flat_v[untouched].any()
    # slot 16 is block 1, row 0 of the [num_blocks, block_size, ...] cache
    np.testing.assert_array_equal(kc[1, 0], key[2])


def test_store_random_slots_matches_numpy_scatter():
    rng = np.random.default_rng(3)
    nb, bs, hkv, d, T = 12, 16, 4, 64, 70
    slots = rng.permutation(nb * bs)[:T].astype(np.int32)
    slots[rng.random(T) < 0.2] = -1
    key = rng.integers(0, 1 << 16, (T, hkv, d), dtype=np.uint16)
    value = rng.integers(0, 1 << 16, (T, hkv, d), dtype=np.uint16)
    kc0 = rng.integers(0, 1 << 16, (nb, bs, hkv, d), dtype=np.uint16)
    vc0 = rng.integers(0, 1 << 16, (nb, bs, hkv, d), dtype=np.uint16)
    kc, vc = kc0.copy(), vc0.copy()
    oracle.store_kvcache(key, value, kc, vc, slots, bs)
    ek, ev = kc0.reshape(nb * bs, hkv, d).copy(), vc0.reshape(nb * bs, hkv, d).copy()
    keep = slots >= 0
    ek[slots[keep]] = key[keep]
    ev[slots[keep]] = value[keep]
    np.testing.assert_array_equal(kc.reshape(nb * bs, hkv, d), ek)
    np.testing.assert_array_equal(vc.reshape(nb * bs, hkv, d), ev)


def test_store_rejects_slot_past_the_pool():
    kc = np.zeros((2, 16, 1, 8), np.uint16)
    with pytest.raises(oracle.OracleError):
        oracle.store_kvcache(np.zeros((1, 1, 8), np.uint16), np.zeros((1, 1, 8), np.uint16),
                             kc, kc.copy(), np.array([32], np.int32), 16)


def test_bf16_widening_is_exact():
    for bits, val in ((0x3F80, 1.0), (0xC000, -2.0), (0x3E80, 0.25), (0x0000, 0.0),
                      (0x7F80, math.inf)):
        assert oracle.bf16_to_double(bits) == val


# -------------------------------------------------------------- attention ---

def _contiguous_case(H, Hkv, D, ctx, ql, window=0, bs=16, seed=0):
    """A case whose block tables are the identity (sequence i owns consecutive blocks
    in pool order), so the paged cache read equals a contiguous K/V per sequence."""
    w = Workload("pin", H, Hkv, D, bs, (), sliding_window=window)
    case = make_case_from_lengths(w, ctx, ql, seed=seed)
    nblk = (case.seq_lens + bs - 1) // bs
    bt = np.full_like(case.block_table, -1)
    c = 0
    for i, n in enumerate(nblk):
        bt[i, :n] = np.arange(c, c + n)
        c += n
    case.block_table = bt
    return case


def _run_oracle(case, window=None, num_threads=0):
    w = case.workload
    return oracle.paged_attention(bf16_bits(case.q), bf16_bits(case.k_cache),
                                  bf16_bits(case.v_cache), case.cu_seqlens_q, case.seq_lens,
                                  case.block_table, w.num_heads, w.num_kv_heads,
                                  w.sliding_window if window is None else window,
                                  w.final_scale, num_threads)


def _contiguous_kv(case, i):
    """K, V [sk, Hkv, D] float64 of sequence i read straight from the pool order."""
    bs = case.workload.block_size
    sk = int(case.seq_lens[i])
    blocks = case.block_table[i, :(sk + bs - 1) // bs]
    k = case.k_cache.double()[torch.as_tensor(blocks, dtype=torch.long)].reshape(
        -1, case.workload.num_kv_heads, case.workload.head_dim)[:sk]
    v = case.v_cache.double()[torch.as_tensor(blocks, dtype=torch.long)].reshape(
        -1, case.workload.num_kv_heads, case.workload.head_dim)[:sk]
    return k, v


@pytest.mark.parametrize("H,Hkv", [(4, 4), (8, 2), (10, 2)])
def test_prefill_equals_torch_sdpa_causal(H, Hkv):
    # torch_sdpa.py prompt path: per-sequence scaled_dot_product_attention with
    # is_causal and K/V repeat_interleave'd by num_queries_per_kv.
    case = _contiguous_case(H, Hkv, 32, [0, 0, 0], [5, 17, 33], seed=1)
    got = _run_oracle(case)
    G = H // Hkv
    for i in range(case.num_seqs):
        a, b = case.cu_seqlens_q[i], case.cu_seqlens_q[i + 1]
        q = case.q[a:b].double().transpose(0, 1)
        k, v = _contiguous_kv(case, i)
        k = k.repeat_interleave(G, dim=1).transpose(0, 1)
        v = v.repeat_interleave(G, dim=1).transpose(0, 1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, is_causal=True, scale=case.workload.final_scale).transpose(0, 1)
        np.testing.assert_allclose(got[a:b], ref.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("window", [0, 1, 3, 16, 40])
def test_chunked_prefill_equals_sdpa_with_hf_mask(window):
    case = _contiguous_case(8, 2, 64, [0, 9, 30, 47], [6, 7, 1, 20], window=window, seed=2)
    got = _run_oracle(case)
    for i in range(case.num_seqs):
        a, b = case.cu_seqlens_q[i], case.cu_seqlens_q[i + 1]
        sq, sk = b - a, int(case.seq_lens[i])
        if window == 1:  # HF spells "no window" as 1; the square sdpa formula covers w = 1
            ones = torch.ones(sq, sk)
            allowed = torch.zeros(sq, sk, dtype=torch.bool)
            for r in range(sq):
                allowed[r, sk - sq + r] = True
        else:
            allowed = torch.as_tensor(_hf_formula_allowed(sq, sk, window))
        q = case.q[a:b].double().transpose(0, 1)
        k, v = _contiguous_kv(case, i)
        k = k.repeat_interleave(4, dim=1).transpose(0, 1)
        v = v.repeat_interleave(4, dim=1).transpose(0, 1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, attn_mask=allowed, scale=case.workload.final_scale).transpose(0, 1)
        np.testing.assert_allclose(got[a:b], ref.numpy(), rtol=0, atol=1e-12)


def test_block_table_permutation_invariance():
    case = make_case("batched_decode_small", seed=5)
    base = _run_oracle(case)
    rng = np.random.default_rng(0)
    nb = case.num_blocks
    perm = rng.permutation(nb)  # new physical index of old block b is perm[b]
    kc = torch.empty_like(case.k_cache)
    vc = torch.empty_like(case.v_cache)
    kc[torch.as_tensor(perm)] = case.k_cache
    vc[torch.as_tensor(perm)] = case.v_cache
    bt = np.where(case.block_table >= 0, perm[np.maximum(case.block_table, 0)], -1)
    case.k_cache, case.v_cache, case.block_table = kc, vc, bt.astype(np.int32)
    np.testing.assert_array_equal(_run_oracle(case), base)


def test_constant_v_gives_v():
    case = make_case("mixed_window_small", seed=6)
    row = torch.randn(case.workload.num_kv_heads, case.workload.head_dim).to(torch.bfloat16)
    case.v_cache[:] = row
    got = _run_oracle(case)
    G = case.workload.num_heads // case.workload.num_kv_heads
    expect = row.double().repeat_interleave(G, dim=0).numpy()
    np.testing.assert_allclose(got, np.broadcast_to(expect, got.shape), rtol=0, atol=1e-12)


def test_zero_query_gives_mean_of_visible_values():
    # q = 0 -> every visible logit is 0 -> uniform weights (closed form).
    case = make_case("mixed_window_small", seed=8)
    case.q.zero_()
    got = _run_oracle(case)
    w = case.workload
    G = w.num_heads // w.num_kv_heads
    for i in range(case.num_seqs):
        k, v = _contiguous_kv_any(case, i)
        a = case.cu_seqlens_q[i]
        sq, sk = case.query_lens[i], case.seq_lens[i]
        for r in (0, sq - 1):
            p = sk - sq + r
            lo = max(0, p - w.sliding_window + 1) if w.sliding_window > 0 else 0
            mean = v[lo:p + 1].mean(0)
            np.testing.assert_allclose(got[a + r], mean.repeat_interleave(G, 0).numpy(),
                                       rtol=0, atol=1e-12)


def _contiguous_kv_any(case, i):
    bs = case.workload.block_size
    sk = int(case.seq_lens[i])
    idx = torch.as_tensor(case.block_table[i, :(sk + bs - 1) // bs], dtype=torch.long)
    shp = (-1, case.workload.num_kv_heads, case.workload.head_dim)
    return (case.k_cache.double()[idx].reshape(shp)[:sk],
            case.v_cache.double()[idx].reshape(shp)[:sk])


def test_decode_equals_last_row_of_full_prefill():
    w = Workload("pin", 8, 2, 64, 16, ())
    lens = [1, 16, 17, 50]
    pre = make_case_from_lengths(w, [0] * 4, lens, seed=9)
    full = _run_oracle(pre)
    dec = make_case_from_lengths(w, [n - 1 for n in lens], [1] * 4, seed=9)
    dec.k_cache, dec.v_cache, dec.block_table = pre.k_cache, pre.v_cache, pre.block_table
    dec.q = pre.q[torch.as_tensor(pre.cu_seqlens_q[1:] - 1, dtype=torch.long)]
    got = _run_oracle(dec)
    np.testing.assert_array_equal(got, full[pre.cu_seqlens_q[1:] - 1])


def test_gqa_equals_mha_with_repeated_kv_heads():
    case = make_case("mixed_window_small", seed=10)
    gqa = _run_oracle(case)
    w = case.workload
    G = w.num_heads // w.num_kv_heads
    mha_w = Workload("mha", w.num_heads, w.num_heads, w.head_dim, w.block_size, (),
                     sliding_window=w.sliding_window)
    mha = make_case_from_lengths(mha_w, case.context_lens, case.query_lens, seed=10)
    mha.q = case.q
    mha.block_table = case.block_table
    mha.k_cache = case.k_cache.repeat_interleave(G, dim=2).contiguous()
    mha.v_cache = case.v_cache.repeat_interleave(G, dim=2).contiguous()
    np.testing.assert_array_equal(_run_oracle(mha), gqa)


def test_window_at_least_seq_len_is_no_window_and_window_one_is_own_value():
    case = make_case("mixed_window_small", seed=11)
    big = int(case.seq_lens.max())
    np.testing.assert_array_equal(_run_oracle(case, window=big), _run_oracle(case, window=0))
    got = _run_oracle(case, window=1)
    w = case.workload
    G = w.num_heads // w.num_kv_heads
    for i in range(case.num_seqs):
        _, v = _contiguous_kv_any(case, i)
        a = case.cu_seqlens_q[i]
        sq, sk = case.query_lens[i], case.seq_lens[i]
        for r in range(sq):
            np.testing.assert_array_equal(
                got[a + r], v[sk - sq + r].repeat_interleave(G, 0).numpy())


def test_brute_force_tiny_against_hand_softmax():
    # Two keys, one head: o = (e^{s0} v0 + e^{s1} v1) / (e^{s0} + e^{s1}).
    w = Workload("pin", 1, 1, 8, 1, (), scale=0.5)
    case = make_case_from_lengths(w, [1], [1], seed=12)
    got = _run_oracle(case)[0, 0]
    q = case.q.double()[0, 0]
    ks = [case.k_cache.double()[case.block_table[0, j], 0, 0] for j in range(2)]
    vs = [case.v_cache.double()[case.block_table[0, j], 0, 0] for j in range(2)]
    s = [0.5 * float(q @ k) for k in ks]
    e = [math.exp(x) for x in s]
    expect = (e[0] * vs[0] + e[1] * vs[1]) / (e[0] + e[1])
    np.testing.assert_allclose(got, expect.numpy(), rtol=1e-14, atol=1e-14)


def test_empty_sequence_gives_zero_row_and_bad_block_is_reported():
    w = Workload("pin", 2, 1, 16, 16, ())
    case = make_case_from_lengths(w, [0, 3], [0, 1], seed=13)
    # decode-style call with an empty first sequence
    out = oracle.paged_attention(bf16_bits(case.q), bf16_bits(case.k_cache),
                                 bf16_bits(case.v_cache), np.array([0, 0, 1], np.int32),
                                 case.seq_lens, case.block_table, 2, 1, 0, 0.25)
    assert out.shape[0] == 1
    bad = case.block_table.copy()
    bad[1, 0] = case.num_blocks + 5
    with pytest.raises(oracle.OracleError):
        oracle.paged_attention(bf16_bits(case.q), bf16_bits(case.k_cache),
                               bf16_bits(case.v_cache), case.cu_seqlens_q, case.seq_lens, bad,
                               2, 1, 0, 0.25)
    row = oracle.attend_row(bf16_bits(case.q[0]), bf16_bits(case.k_cache),
                            bf16_bits(case.v_cache), case.block_table[0], 0, 0, 2, 1, 0, 0.25)
    assert not row.any()


def test_thread_count_does_not_change_result():
    case = make_case("varlen_prefill_small", seed=14)
    np.testing.assert_array_equal(_run_oracle(case, num_threads=1), _run_oracle(case, num_threads=5))


# ------------------------------------------------------- partial results (state) ---
# "05 Attention Backends", section 7.1 (split-KV) and section 8 (cascade): attention over
# a key set may be computed per disjoint part and merged; these pins tie the oracle's
# state and merge to the plain attention pinned above.

def _state(case, i, key_begin, window=0):
    w = case.workload
    sk = int(case.seq_lens[i])
    return oracle.attend_row_state(bf16_bits(case.q)[case.cu_seqlens_q[i + 1] - 1],
                                   bf16_bits(case.k_cache), bf16_bits(case.v_cache),
                                   case.block_table[i], sk, sk - 1, key_begin, w.num_heads,
                                   w.num_kv_heads, window, w.final_scale)


def _state_range(case, i, begin, end):
    """State of sequence i's last query over keys [begin, end) (no window): a query at
    position end - 1 of the sequence truncated to `end` keys, from key `begin`."""
    w = case.workload
    return oracle.attend_row_state(bf16_bits(case.q)[case.cu_seqlens_q[i + 1] - 1],
                                   bf16_bits(case.k_cache), bf16_bits(case.v_cache),
                                   case.block_table[i], end, end - 1, begin, w.num_heads,
                                   w.num_kv_heads, 0, w.final_scale)


def test_state_of_one_key_is_its_value_and_logit():
    case = _contiguous_case(4, 2, 32, [0], [9], seed=60)
    o, lse = _state(case, 0, key_begin=8)  # only the last key is left
    k, v = _contiguous_kv(case, 0)
    q = case.q.double()[8]
    G = 2
    for h in range(4):
        np.testing.assert_array_equal(o[h], v[8, h // G].numpy())
        logit = case.workload.final_scale * float((q[h] * k[8, h // G]).sum())
        assert lse[h] == pytest.approx(logit, rel=0, abs=1e-12)


@pytest.mark.parametrize("window", [0, 5])
def test_state_of_zero_query_has_lse_log_count(window):
    case = _contiguous_case(4, 4, 16, [0], [23], seed=61)
    case.q.zero_()
    for kb in (0, 7, 22):
        o, lse = _state(case, 0, key_begin=kb, window=window)
        lo = max(kb, 23 - window) if window > 0 else kb
        np.testing.assert_allclose(lse, math.log(23 - lo), rtol=0, atol=1e-12)


def test_merging_disjoint_parts_gives_the_whole():
    w = Workload("st", 8, 2, 32, 16, ())
    case = make_case_from_lengths(w, [0, 0, 0], [70, 33, 130], seed=62)
    for i, cuts in ((0, [1, 40]), (1, [16]), (2, [5, 64, 100])):
        sk = int(case.seq_lens[i])
        whole, whole_lse = _state(case, i, 0)
        edges = [0] + cuts + [sk]
        parts = [_state_range(case, i, a, b) for a, b in zip(edges[:-1], edges[1:])]
        got, got_lse = oracle.merge_states(np.stack([o for o, _ in parts]),
                                           np.stack([l for _, l in parts]))
        np.testing.assert_allclose(got, whole, rtol=0, atol=1e-12)
        np.testing.assert_allclose(got_lse, whole_lse, rtol=0, atol=1e-12)
        # The merge does not depend on the order of the parts.
        got2, _ = oracle.merge_states(np.stack([o for o, _ in parts[::-1]]),
                                      np.stack([l for _, l in parts[::-1]]))
        np.testing.assert_allclose(got2, whole, rtol=0, atol=1e-12)


def test_merge_treats_empty_parts_as_absent():
    rng = np.random.default_rng(63)
    o = rng.standard_normal((1, 5, 8))
    lse = rng.standard_normal((1, 5))
    empty_o, empty_l = np.zeros((1, 5, 8)), np.full((1, 5), -np.inf)
    got, got_lse = oracle.merge_states(np.concatenate([empty_o, o, empty_o]),
                                       np.concatenate([empty_l, lse, empty_l]))
    np.testing.assert_allclose(got, o[0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(got_lse, lse[0], rtol=0, atol=1e-15)
    got, got_lse = oracle.merge_states(np.concatenate([empty_o, empty_o]),
                                       np.concatenate([empty_l, empty_l]))
    assert not got.any() and np.isneginf(got_lse).all()


def test_shared_prefix_attention_is_prefix_state_merged_with_suffix_state():
    # Cascade: sequences whose first P keys live in the same physical blocks.
    w = Workload("cas", 8, 2, 32, 16, ())
    case = make_case_from_lengths(w, [0, 0, 0], [80, 50, 97], seed=64)
    P = 48  # three shared blocks
    case.block_table[1, :3] = case.block_table[0, :3]
    case.block_table[2, :3] = case.block_table[0, :3]
    for i in range(3):
        whole, whole_lse = _state(case, i, 0)
        o1, l1 = _state_range(case, i, 0, P)
        o2, l2 = _state(case, i, P)
        got, got_lse = oracle.merge_states(np.stack([o1, o2]), np.stack([l1, l2]))
        np.testing.assert_allclose(got, whole, rtol=0, atol=1e-12)
        np.testing.assert_allclose(got_lse, whole_lse, rtol=0, atol=1e-12)
    # The prefix state depends only on the shared blocks: same for every sequence
    # whose query is the same.
    case.q[case.cu_seqlens_q[2] - 1] = case.q[case.cu_seqlens_q[1] - 1]
    a, la = _state_range(case, 0, 0, P)
    b, lb = _state_range(case, 1, 0, P)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


# ------------------------------------------------------------------ FP8 E4M3 cache ---
# The E4M3 ("fn") format: sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinities,
# S.1111.111 = NaN, largest finite 448.  Pinned by its defining values, by torch's own
# float8_e4m3fn conversion (a library routine) and by round trips.

def test_fp8_decode_defining_values():
    d = oracle.fp8_e4m3_decode
    assert d(0x38) == 1.0 and d(0x7E) == 448.0 and d(0xFE) == -448.0
    assert d(0x01) == 2.0 ** -9 and d(0x07) == 7 * 2.0 ** -9 and d(0x08) == 2.0 ** -6
    assert d(0x00) == 0.0 and math.copysign(1.0, d(0x80)) == -1.0
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))


def test_fp8_decode_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.fp8_e4m3_decode(c) for c in range(256)])
    finite = ~np.isnan(ref)
    np.testing.assert_array_equal(got[finite], ref[finite])
    assert np.isnan(got[~finite]).all()


def test_fp8_encode_round_trips_and_matches_torch():
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert oracle.fp8_e4m3_encode(oracle.fp8_e4m3_decode(c)) == c
    rng = np.random.default_rng(70)
    xs = np.concatenate([rng.standard_normal(3000) * s for s in (1e-3, 0.1, 1, 30, 200)])
    xs = np.clip(xs, -448, 448).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.fp8_e4m3_encode(x) for x in xs], dtype=np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_fp8_encode_ties_saturation_and_nan():
    e = oracle.fp8_e4m3_encode
    assert e(1.0625) == 0x38 and e(1.1875) == 0x3A    # ties go to the even code
    assert e(1000.0) == 0x7E and e(-1000.0) == 0xFE and e(float("inf")) == 0x7E
    assert e(460.0) == 0x7E                             # between 448 and the next grid point
    assert e(float("nan")) == 0x7F


def test_fp8_store_quantises_x_over_scale():
    w = Workload("f8", 4, 2, 16, 16, ())
    case = make_case_from_lengths(w, [0], [5], seed=71)
    kc = np.zeros((case.k_cache.shape[0], 16, 2, 16), dtype=np.uint8)
    vc = np.zeros_like(kc)
    oracle.store_kvcache_fp8(bf16_bits(case.key), bf16_bits(case.value), kc, vc,
                             case.slot_mapping, 16, 0.25)
    k = case.key.float().numpy()
    for t, slot in enumerate(case.slot_mapping):
        blk, off = divmod(int(slot), 16)
        want = (torch.from_numpy((k[t] / np.float32(0.25)).astype(np.float32))
                .to(torch.float8_e4m3fn).view(torch.uint8).numpy())
        np.testing.assert_array_equal(kc[blk, off], want)


def test_fp8_attention_equals_bf16_attention_on_exact_values():
    # Cache values that are E4M3 codes times kv_scale and also exact bf16: both oracle
    # paths must give the same result.
    w = Workload("f8a", 8, 2, 32, 16, ())
    case = make_case_from_lengths(w, [30, 0], [1, 45], seed=72)
    rng = np.random.default_rng(73)
    scale = 0.5
    codes_k = rng.integers(0, 0x7F, size=case.k_cache.shape, dtype=np.uint8) | \
        (rng.integers(0, 2, size=case.k_cache.shape, dtype=np.uint8) << 7)
    codes_v = rng.integers(0, 0x7F, size=case.v_cache.shape, dtype=np.uint8)
    vals_k = np.vectorize(oracle.fp8_e4m3_decode)(codes_k) * scale
    vals_v = np.vectorize(oracle.fp8_e4m3_decode)(codes_v) * scale
    kb = torch.from_numpy(vals_k).to(torch.bfloat16)
    vb = torch.from_numpy(vals_v).to(torch.bfloat16)
    assert np.array_equal(kb.double().numpy(), vals_k)  # exact in bf16
    ref = oracle.paged_attention(bf16_bits(case.q), bf16_bits(kb), bf16_bits(vb),
                                 case.cu_seqlens_q, case.seq_lens, case.block_table, 8, 2, 0,
                                 w.final_scale)
    got = oracle.paged_attention_fp8(bf16_bits(case.q), codes_k, codes_v, case.cu_seqlens_q,
                                     case.seq_lens, case.block_table, 8, 2, 0, w.final_scale,
                                     scale)
    np.testing.assert_array_equal(got, ref)
