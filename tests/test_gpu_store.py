"""pa_store_kvcache on the GPU: bit-exact against the oracle's store."""
import os

import numpy as np
import pytest
import torch

import paged_kv_attention_03_gb300 as pa
from paged_kv_attention_03_gb300.inputs import (SMALL_WORKLOADS, WORKLOADS, Workload,
                                                bf16_bits, make_case, make_case_from_lengths)

from _parity import device_tensors, host_inputs, oracle_store

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _check_store(case, dev):
    h = host_inputs(case)
    oracle_store(case, h)
    m = device_tensors(case, dev)
    pa.pa_store_kvcache(case.key, case.value, case.k_cache, case.v_cache, m["slot_mapping"])
    assert pa.pa_read_device_error(device=dev) == 0
    np.testing.assert_array_equal(bf16_bits(case.k_cache), h["k_cache"])
    np.testing.assert_array_equal(bf16_bits(case.v_cache), h["v_cache"])


def test_store_printed_example(cuda):
    # "MinivLLM API docs - Attention", store_kvcache example: slots [0, 1, 16, -1].
    g = torch.Generator().manual_seed(7)
    key = torch.randn(4, 2, 64, generator=g).to(torch.bfloat16).to(cuda)
    value = torch.randn(4, 2, 64, generator=g).to(torch.bfloat16).to(cuda)
    kc = torch.zeros(8, 16, 2, 64, dtype=torch.bfloat16, device=cuda)
    vc = torch.zeros_like(kc)
    slots = torch.tensor([0, 1, 16, -1], dtype=torch.int32, device=cuda)
    pa.pa_store_kvcache(key, value, kc, vc, slots)
    fk, fv = kc.view(128, 2, 64).cpu(), vc.view(128, 2, 64).cpu()
    for t, s in ((0, 0), (1, 1), (2, 16)):
        assert torch.equal(fk[s], key[t].cpu()) and torch.equal(fv[s], value[t].cpu())
    mask = torch.ones(128, dtype=torch.bool)
    mask[[0, 1, 16]] = False
    assert not fk[mask].any() and not fv[mask].any()


@pytest.mark.parametrize("name", list(SMALL_WORKLOADS))
def test_store_small_workloads(cuda, name):
    _check_store(make_case(name, seed=21, device=cuda), cuda)


@pytest.mark.parametrize("name", ["varlen_prefill", "batched_decode", "mixed_window"])
def test_store_full_size_workloads(cuda, name):
    _check_store(make_case(name, seed=22, device=cuda), cuda)


@pytest.mark.parametrize("hkv,d", [(1, 64), (2, 128), (8, 128), (3, 64)])
def test_store_padding_and_odd_rows(cuda, hkv, d):
    w = Workload("store", hkv, hkv, d, 16, ())
    case = make_case_from_lengths(w, [5, 0, 37], [9, 1, 30], seed=23, device=cuda)
    rng = np.random.default_rng(1)
    case.slot_mapping[rng.random(case.slot_mapping.shape[0]) < 0.3] = -1
    _check_store(case, cuda)


def test_store_out_of_range_slot_is_flagged_and_skipped(cuda):
    w = Workload("store", 2, 2, 64, 16, ())
    case = make_case_from_lengths(w, [0, 0], [3, 2], seed=24, device=cuda)
    bad = case.slot_mapping.copy()
    bad[1] = case.num_blocks * 16 + 3  # past the pool
    case.slot_mapping = bad.copy()
    h = host_inputs(case)
    keep = bad.copy()
    keep[1] = -1
    import oracle
    oracle.store_kvcache(h["key"], h["value"], h["k_cache"], h["v_cache"], keep, 16)
    slots = torch.as_tensor(bad, device=cuda)
    pa.pa_store_kvcache(case.key, case.value, case.k_cache, case.v_cache, slots)
    assert pa.pa_read_device_error(device=cuda) & pa.DEVERR_SLOT_RANGE
    np.testing.assert_array_equal(bf16_bits(case.k_cache), h["k_cache"])
    assert pa.pa_read_device_error(device=cuda) == 0  # cleared


def test_store_empty_is_noop(cuda):
    kc = torch.zeros(2, 16, 1, 64, dtype=torch.bfloat16, device=cuda)
    e = torch.empty(0, 1, 64, dtype=torch.bfloat16, device=cuda)
    pa.pa_store_kvcache(e, e, kc, kc.clone(), torch.empty(0, dtype=torch.int32, device=cuda))
    assert not kc.any()
