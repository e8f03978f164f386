"""Device-side failure detection of the prefill kernel: a wait that runs out raises
PA_DEVERR_TIMEOUT and the kernel returns, leaving the device usable.

The testing aid pa_debug_prefill_stall makes the kernel hand out no work item, so
every role's first wait runs out while no copy or product is in flight; the wait limit
is lowered to 20 ms for the test.
"""
import numpy as np
import pytest

import paged_kv_attention_03_gb300 as pa
from paged_kv_attention_03_gb300.inputs import make_case

from _parity import assert_parity, device_tensors, host_inputs, oracle_attention, oracle_store

pytestmark = pytest.mark.gpu


def _run_prefill(case, dev, **kw):
    w = case.workload
    m = device_tensors(case, dev)
    return pa.pa_varlen_prefill(case.q, case.k_cache, case.v_cache, m["cu_seqlens_q"],
                                m["seq_lens"], m["block_table"], case.max_query_len,
                                case.max_seq_len, w.final_scale, w.sliding_window, **kw)


def test_prefill_wait_limit_runs_out_then_device_is_usable(cuda):
    case = make_case("varlen_prefill_small", seed=60, device=cuda)
    pa.pa_read_device_error(clear=True, device=cuda)
    pa.pa_debug_prefill_stall(True, 20_000_000)
    try:
        _run_prefill(case, cuda)
        flags = pa.pa_read_device_error(clear=True, device=cuda)
    finally:
        pa.pa_debug_prefill_stall(False, 0)
    assert flags & pa.DEVERR_TIMEOUT, f"flags {flags:#x}"
    # The same device and process run a normal call with parity: the stalled launch
    # freed its tensor memory and left no fault behind.
    h = host_inputs(case)
    oracle_store(case, h)
    m = device_tensors(case, cuda)
    out = _run_prefill(case, cuda, key=case.key, value=case.value,
                       slot_mapping=m["slot_mapping"])
    assert pa.pa_read_device_error(clear=True, device=cuda) == 0
    assert_parity(out, oracle_attention(case, h), "after a timed-out launch")


def test_cascade_prefix_wait_limit_runs_out_then_device_is_usable(cuda):
    from paged_kv_attention_03_gb300.inputs import Workload, make_shared_prefix_case
    import torch
    w = Workload("shared_prefix", 32, 8, 128, 16, ())
    case = make_shared_prefix_case(w, 8, np.array([5, 40, 17]), 61, cuda)
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=cuda)
    bt, sl = t(case.block_table), t(case.seq_lens)
    max_len = int(case.seq_lens.max())
    pa.pa_read_device_error(clear=True, device=cuda)
    pa.pa_debug_prefill_stall(True, 20_000_000)
    try:
        pa.pa_cascade_decode(case.q, case.k_cache, case.v_cache, bt, sl, max_len, 128,
                             w.final_scale, 0)
        flags = pa.pa_read_device_error(clear=True, device=cuda)
    finally:
        pa.pa_debug_prefill_stall(False, 0)
    assert flags & pa.DEVERR_TIMEOUT, f"flags {flags:#x}"
    out = pa.pa_cascade_decode(case.q, case.k_cache, case.v_cache, bt, sl, max_len, 128,
                               w.final_scale, 0)
    assert pa.pa_read_device_error(clear=True, device=cuda) == 0
    h = host_inputs(case)
    assert_parity(out, oracle_attention(case, h), "cascade after a timed-out launch")
