"""FP8 E4M3 KV cache on the GPU against the fp64 oracle.

The store is bit-exact (an integer decision taken in fp32 on both sides: x / kv_scale
correctly rounded, then round to nearest even onto E4M3, saturating at 448).  The
decode reads code * kv_scale exactly and carries the attention bar (max-abs <= 1e-2,
mean-abs <= 1e-3).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_03_gb300 as pa
from paged_kv_attention_03_gb300.inputs import Workload, bf16_bits, make_case_from_lengths

from _parity import assert_parity

pytestmark = pytest.mark.gpu


def _t(a, dev):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=dev)


def _codes_of(cache_bf16, kv_scale):
    """E4M3 codes of the N(0,1) bf16 cache / kv_scale (test input, as a store would give)."""
    return (cache_bf16.float().cpu() / kv_scale).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("kv_scale", [0.5, 0.03])
def test_fp8_store_is_bit_exact(cuda, kv_scale):
    w = Workload("s8", 8, 4, 128, 16, ())
    case = make_case_from_lengths(w, [0, 10], [300, 77], seed=100, device=cuda)
    # Spread magnitudes: subnormal range, normal range, ties and saturation (|x| > 448 s).
    g = torch.Generator(device="cpu").manual_seed(101)
    mags = torch.tensor([1e-4, 1e-2, 1.0, 20.0, 1000.0])
    pick = torch.randint(0, 5, case.key.shape, generator=g)
    case.key.copy_((torch.randn(case.key.shape, generator=g) * mags[pick]).to(torch.bfloat16))
    case.value.copy_((torch.randn(case.value.shape, generator=g) * mags[pick]).to(torch.bfloat16))
    kc = torch.zeros(case.k_cache.shape, dtype=torch.uint8, device=cuda)
    vc = torch.zeros_like(kc)
    pa.pa_store_kvcache_fp8(case.key, case.value, kc, vc, _t(case.slot_mapping, cuda), kv_scale)
    assert pa.pa_read_device_error(device=cuda) == 0
    hk = np.zeros(kc.shape, np.uint8)
    hv = np.zeros(vc.shape, np.uint8)
    oracle.store_kvcache_fp8(bf16_bits(case.key), bf16_bits(case.value), hk, hv,
                             case.slot_mapping, 16, kv_scale)
    np.testing.assert_array_equal(kc.cpu().numpy(), hk)
    np.testing.assert_array_equal(vc.cpu().numpy(), hv)


def _fp8_case(dev, H, Hkv, D, lens, bs=16, seed=102, kv_scale=0.02):
    w = Workload("d8", H, Hkv, D, bs, ())
    case = make_case_from_lengths(w, [n - 1 for n in lens], [1] * len(lens), seed=seed,
                                  device=dev)
    return case, _codes_of(case.k_cache, kv_scale), _codes_of(case.v_cache, kv_scale), kv_scale


@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("window", [0, 100])
def test_fp8_decode_matches_oracle(cuda, splits, window):
    case, kc, vc, s = _fp8_case(cuda, 32, 8, 128, [1, 17, 500, 2048, 3000])
    out = pa.pa_decode_fp8(case.q, torch.from_numpy(kc).to(cuda), torch.from_numpy(vc).to(cuda),
                           _t(case.block_table, cuda), _t(case.seq_lens, cuda),
                           int(case.seq_lens.max()), case.workload.final_scale, s, window,
                           splits)
    assert pa.pa_read_device_error(device=cuda) == 0
    ref = oracle.paged_attention_fp8(bf16_bits(case.q), kc, vc, case.cu_seqlens_q,
                                     case.seq_lens, case.block_table, 32, 8, window,
                                     case.workload.final_scale, s)
    assert_parity(out, ref, f"fp8 decode splits={splits} window={window}")


@pytest.mark.parametrize("H,Hkv,D,bs", [(40, 8, 128, 16), (8, 8, 64, 32), (16, 2, 128, 8),
                                        (24, 2, 64, 16), (32, 2, 128, 16), (20, 1, 128, 16)])
def test_fp8_decode_shapes(cuda, H, Hkv, D, bs):
    case, kc, vc, s = _fp8_case(cuda, H, Hkv, D, [5, 64, 333], bs=bs, seed=103, kv_scale=0.1)
    out = pa.pa_decode_fp8(case.q, torch.from_numpy(kc).to(cuda), torch.from_numpy(vc).to(cuda),
                           _t(case.block_table, cuda), _t(case.seq_lens, cuda),
                           int(case.seq_lens.max()), case.workload.final_scale, s)
    ref = oracle.paged_attention_fp8(bf16_bits(case.q), kc, vc, case.cu_seqlens_q,
                                     case.seq_lens, case.block_table, H, Hkv, 0,
                                     case.workload.final_scale, s)
    assert_parity(out, ref, f"fp8 {H}/{Hkv} D={D} bs={bs}")


def test_fp8_decode_with_fused_store(cuda):
    case, kc, vc, s = _fp8_case(cuda, 32, 8, 128, [40, 700, 1], seed=104, kv_scale=0.05)
    hk, hv = kc.copy(), vc.copy()
    oracle.store_kvcache_fp8(bf16_bits(case.key), bf16_bits(case.value), hk, hv,
                             case.slot_mapping, 16, s)
    dk, dv = torch.from_numpy(kc).to(cuda), torch.from_numpy(vc).to(cuda)
    out = pa.pa_decode_fp8(case.q, dk, dv, _t(case.block_table, cuda), _t(case.seq_lens, cuda),
                           int(case.seq_lens.max()), case.workload.final_scale, s,
                           key=case.key, value=case.value,
                           slot_mapping=_t(case.slot_mapping, cuda))
    assert pa.pa_read_device_error(device=cuda) == 0
    np.testing.assert_array_equal(dk.cpu().numpy(), hk)
    np.testing.assert_array_equal(dv.cpu().numpy(), hv)
    ref = oracle.paged_attention_fp8(bf16_bits(case.q), hk, hv, case.cu_seqlens_q,
                                     case.seq_lens, case.block_table, 32, 8, 0,
                                     case.workload.final_scale, s)
    assert_parity(out, ref, "fp8 fused store")


# ----------------------------------------------------------------- varlen prefill ---

def _fp8_prefill_case(dev, ctx, qlens, H=32, Hkv=8, bs=16, seed=110, kv_scale=0.02):
    w = Workload("p8", H, Hkv, 128, bs, ())
    case = make_case_from_lengths(w, ctx, qlens, seed=seed, device=dev)
    return case, _codes_of(case.k_cache, kv_scale), _codes_of(case.v_cache, kv_scale), kv_scale


def _fp8_prefill_check(case, kc, vc, s, dev, window=0, fused_store=False, what=""):
    """pa_varlen_prefill_fp8 over the codes (optionally storing the step's tokens first)
    against the FP8 oracle on every row."""
    hk, hv = kc.copy(), vc.copy()
    kw = {}
    if fused_store:
        oracle.store_kvcache_fp8(bf16_bits(case.key), bf16_bits(case.value), hk, hv,
                                 case.slot_mapping, case.workload.block_size, s)
        kw = dict(key=case.key, value=case.value, slot_mapping=_t(case.slot_mapping, dev))
    dk, dv = torch.from_numpy(kc).to(dev), torch.from_numpy(vc).to(dev)
    w = case.workload
    out = pa.pa_varlen_prefill_fp8(case.q, dk, dv, _t(case.cu_seqlens_q, dev),
                                   _t(case.seq_lens, dev), _t(case.block_table, dev),
                                   case.max_query_len, case.max_seq_len, w.final_scale, s,
                                   window, **kw)
    flags = pa.pa_read_device_error(device=dev)
    assert flags == 0, f"device error bits {flags:#x}"
    if fused_store:
        np.testing.assert_array_equal(dk.cpu().numpy(), hk)
        np.testing.assert_array_equal(dv.cpu().numpy(), hv)
    ref = oracle.paged_attention_fp8(bf16_bits(case.q), hk, hv, case.cu_seqlens_q,
                                     case.seq_lens, case.block_table, w.num_heads,
                                     w.num_kv_heads, window, w.final_scale, s)
    return assert_parity(out, ref, what or f"fp8 prefill window={window}")


@pytest.mark.parametrize("window", [0, 1, 100, 300])
def test_fp8_prefill_windows_and_chunks(cuda, window):
    case, kc, vc, s = _fp8_prefill_case(cuda, [0, 0, 37, 130, 500, 3], [1, 160, 64, 129, 31, 1])
    _fp8_prefill_check(case, kc, vc, s, cuda, window=window)


@pytest.mark.parametrize("lens", [[16], [127], [128], [129], [255], [257], [700]])
def test_fp8_prefill_tile_edges(cuda, lens):
    case, kc, vc, s = _fp8_prefill_case(cuda, [0] * len(lens), lens, seed=111, kv_scale=0.5)
    _fp8_prefill_check(case, kc, vc, s, cuda)


@pytest.mark.parametrize("H,Hkv,bs", [(8, 8, 16), (40, 8, 32), (16, 2, 64), (64, 4, 256)])
def test_fp8_prefill_shapes(cuda, H, Hkv, bs):
    case, kc, vc, s = _fp8_prefill_case(cuda, [0, 5, 100], [150, 17, 33], H=H, Hkv=Hkv, bs=bs,
                                        seed=112, kv_scale=0.1)
    _fp8_prefill_check(case, kc, vc, s, cuda)
    _fp8_prefill_check(case, kc, vc, s, cuda, window=50)


def test_fp8_prefill_many_sequences(cuda):
    rng = np.random.default_rng(8)
    q = rng.integers(1, 301, size=150)
    ctx = np.where(rng.random(150) < 0.3, rng.integers(0, 200, size=150), 0)
    case, kc, vc, s = _fp8_prefill_case(cuda, ctx, q, seed=113)
    _fp8_prefill_check(case, kc, vc, s, cuda)


def test_fp8_mixed_batch_with_store(cuda):
    # Chunks with a cached context and single-row decodes in one call over an FP8 cache; the
    # call quantises the step's new tokens into the cache first.
    case, kc, vc, s = _fp8_prefill_case(cuda, [1000, 0, 37, 4000, 9, 600],
                                        [512, 300, 1, 1, 1, 200], seed=114, kv_scale=0.05)
    _fp8_prefill_check(case, kc, vc, s, cuda, window=0, fused_store=True, what="fp8 mixed")
    _fp8_prefill_check(case, kc, vc, s, cuda, window=700, fused_store=True,
                       what="fp8 mixed window")


def test_fp8_prefill_rejects_head_dim_64(cuda):
    w = Workload("p8d64", 8, 2, 64, 16, ())
    case = make_case_from_lengths(w, [0], [40], seed=115, device=cuda)
    kc = torch.zeros(case.k_cache.shape, dtype=torch.uint8, device=cuda)
    with pytest.raises(pa.PAError) as e:
        pa.pa_varlen_prefill_fp8(case.q, kc, kc.clone(), _t(case.cu_seqlens_q, cuda),
                                 _t(case.seq_lens, cuda), _t(case.block_table, cuda), 40, 40,
                                 w.final_scale, 0.1)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED


def test_fp8_prefill_full_size_varlen(cuda):
    # The varlen-prefill workload (16 prompts of U[128, 2048], 32/8 heads) over an E4M3 cache
    # holding codes of the N(0,1) pool / 0.02; the step's tokens quantised by the call.
    from paged_kv_attention_03_gb300.inputs import make_case
    case = make_case("varlen_prefill", seed=0, device=cuda)
    s = 0.02
    kc, vc = _codes_of(case.k_cache, s), _codes_of(case.v_cache, s)
    _fp8_prefill_check(case, kc, vc, s, cuda, fused_store=True,
                       what="full size varlen_prefill over an FP8 cache")


def test_fp8_prefill_wait_limit_runs_out_then_device_is_usable(cuda):
    # The FP8 K / V producers poll instead of waiting on one barrier; with the testing aid
    # (no work item handed out) their idle spell and every other role's wait run out after
    # 20 ms, the launch flags PA_DEVERR_TIMEOUT and returns, and the next call is correct.
    case, kc, vc, s = _fp8_prefill_case(cuda, [0, 30], [200, 64], seed=116)
    w = case.workload
    pa.pa_read_device_error(clear=True, device=cuda)
    pa.pa_debug_prefill_stall(True, 20_000_000)
    try:
        pa.pa_varlen_prefill_fp8(case.q, torch.from_numpy(kc).to(cuda),
                                 torch.from_numpy(vc).to(cuda), _t(case.cu_seqlens_q, cuda),
                                 _t(case.seq_lens, cuda), _t(case.block_table, cuda),
                                 case.max_query_len, case.max_seq_len, w.final_scale, s, 0)
        flags = pa.pa_read_device_error(clear=True, device=cuda)
    finally:
        pa.pa_debug_prefill_stall(False, 0)
    assert flags & pa.DEVERR_TIMEOUT, f"flags {flags:#x}"
    _fp8_prefill_check(case, kc, vc, s, cuda, what="FP8 prefill after a timed-out launch")
