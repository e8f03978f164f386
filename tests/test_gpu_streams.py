"""Calls issued on a stream other than the default one.

The C ABI takes the stream as an argument and the binding passes the caller's current
stream: every launch of a call (the store, the split kernel and its combine, the prefill
kernel and the decode launch beside it) must be ordered on that stream.  Each test queues
a long sleep, then a NaN fill of the output, then the call, then a snapshot on a side
stream, with no synchronisation in between: a launch that went to another stream would
run during the sleep and its result would be overwritten by the fill.
"""
import pytest
import torch

import paged_kv_attention_03_gb300 as pa
from paged_kv_attention_03_gb300.inputs import Workload, make_case_from_lengths

from _parity import device_tensors

pytestmark = pytest.mark.gpu

_SLEEP_CYCLES = 50_000_000  # ~25 ms at 2 GHz


def _on_side_stream(call, out):
    """Run `call` on a side stream behind a sleep and a NaN fill of `out`; return the
    snapshot of `out` taken on that stream right after the call."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        torch.cuda._sleep(_SLEEP_CYCLES)
        out.fill_(float("nan"))
        call()
        snap = out.clone()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    return snap


@pytest.mark.parametrize("splits", [1, 0])
def test_decode_on_a_side_stream(cuda, splits):
    w = Workload("sd", 32, 8, 128, 16, ())
    case = make_case_from_lengths(w, [0, 15, 700, 2047, 3000], [1] * 5, seed=93, device=cuda)
    m = device_tensors(case, cuda)
    max_len = int(case.seq_lens.max())
    out = torch.empty_like(case.q)

    def call():
        pa.pa_decode(case.q, case.k_cache, case.v_cache, m["block_table"], m["seq_lens"],
                     max_len, w.final_scale, 0, splits, key=case.key, value=case.value,
                     slot_mapping=m["slot_mapping"], out=out)

    snap = _on_side_stream(call, out)
    ref = torch.empty_like(out)
    pa.pa_decode(case.q, case.k_cache, case.v_cache, m["block_table"], m["seq_lens"], max_len,
                 w.final_scale, 0, splits, key=case.key, value=case.value,
                 slot_mapping=m["slot_mapping"], out=ref)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error(device=cuda) == 0
    assert torch.equal(snap, ref)


def test_mixed_prefill_on_a_side_stream(cuda):
    w = Workload("sp", 32, 8, 128, 16, ())
    case = make_case_from_lengths(w, [0, 5, 300, 1000], [200, 1, 129, 1], seed=94, device=cuda)
    m = device_tensors(case, cuda)
    out = torch.empty_like(case.q)

    def call(dst):
        pa.pa_varlen_prefill(case.q, case.k_cache, case.v_cache, m["cu_seqlens_q"],
                             m["seq_lens"], m["block_table"], case.max_query_len,
                             case.max_seq_len, w.final_scale, 0, key=case.key,
                             value=case.value, slot_mapping=m["slot_mapping"], out=dst)

    snap = _on_side_stream(lambda: call(out), out)
    ref = torch.empty_like(out)
    call(ref)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error(device=cuda) == 0
    assert torch.equal(snap, ref)


def test_store_on_a_side_stream(cuda):
    w = Workload("ss", 8, 2, 64, 16, ())
    case = make_case_from_lengths(w, [3, 40], [20, 7], seed=95, device=cuda)
    m = device_tensors(case, cuda)
    k_ref, v_ref = case.k_cache.clone(), case.v_cache.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        torch.cuda._sleep(_SLEEP_CYCLES)
        case.k_cache.fill_(float("nan"))  # a store on another stream would be overwritten
        case.v_cache.fill_(float("nan"))
        pa.pa_store_kvcache(case.key, case.value, case.k_cache, case.v_cache,
                            m["slot_mapping"])
        k_snap, v_snap = case.k_cache.clone(), case.v_cache.clone()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    k_ref.fill_(float("nan"))
    v_ref.fill_(float("nan"))
    pa.pa_store_kvcache(case.key, case.value, k_ref, v_ref, m["slot_mapping"])
    torch.cuda.synchronize()
    assert pa.pa_read_device_error(device=cuda) == 0
    # NaN != NaN: compare bit patterns.
    assert torch.equal(k_snap.view(torch.int16), k_ref.view(torch.int16))
    assert torch.equal(v_snap.view(torch.int16), v_ref.view(torch.int16))
    # The stored rows hold the new tokens (the rest of the pool keeps the NaN fill).
    slots = m["slot_mapping"].long()
    hkv, d = case.key.shape[1], case.key.shape[2]
    assert torch.equal(k_snap.view(-1, hkv, d)[slots].view(torch.int16), case.key.view(torch.int16))
    assert torch.equal(v_snap.view(-1, hkv, d)[slots].view(torch.int16), case.value.view(torch.int16))


def test_two_calls_on_two_streams_at_once(cuda):
    # A mixed varlen call (its decode launch runs beside the prefill kernel) and a split-K
    # decode with its own workspace, queued on two streams that run at the same time: no
    # state is shared between calls but the device error word.
    wp = Workload("tp", 32, 8, 128, 16, ())
    cp = make_case_from_lengths(wp, [0, 5, 300, 1000], [200, 1, 129, 1], seed=96, device=cuda)
    mp = device_tensors(cp, cuda)
    wd = Workload("td", 32, 8, 128, 16, ())
    cd = make_case_from_lengths(wd, [15, 700, 2047, 3000, 4000], [1] * 5, seed=97, device=cuda)
    md = device_tensors(cd, cuda)
    max_len = int(cd.seq_lens.max())
    ws = torch.empty(max(pa.pa_decode_workspace_size(5, 32, 8, 128, max_len, 0, 0), 1),
                     dtype=torch.uint8, device=cuda)

    def prefill(dst):
        pa.pa_varlen_prefill(cp.q, cp.k_cache, cp.v_cache, mp["cu_seqlens_q"], mp["seq_lens"],
                             mp["block_table"], cp.max_query_len, cp.max_seq_len,
                             wp.final_scale, 0, key=cp.key, value=cp.value,
                             slot_mapping=mp["slot_mapping"], out=dst)

    def decode(dst):
        pa.pa_decode(cd.q, cd.k_cache, cd.v_cache, md["block_table"], md["seq_lens"], max_len,
                     wd.final_scale, 0, 0, key=cd.key, value=cd.value,
                     slot_mapping=md["slot_mapping"], out=dst, workspace=ws)

    out_p, out_d = torch.empty_like(cp.q), torch.empty_like(cd.q)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for s in (s1, s2):
        s.wait_stream(torch.cuda.current_stream())
    for _ in range(3):
        with torch.cuda.stream(s1):
            prefill(out_p)
        with torch.cuda.stream(s2):
            decode(out_d)
    for s in (s1, s2):
        torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref_p, ref_d = torch.empty_like(out_p), torch.empty_like(out_d)
    prefill(ref_p)
    decode(ref_d)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error(device=cuda) == 0
    assert torch.equal(out_p, ref_p)
    assert torch.equal(out_d, ref_d)
