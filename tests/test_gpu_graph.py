"""Attention calls captured in a CUDA graph and replayed.

Serving loops capture their decode step once and replay it: a replay sees only values
held in tensors at fixed addresses ("vllm-npu 0.4.2 wheel diff", xformers.py,
XFormersMetadata, and its use_cuda_graph field for decoding), which is why metadata
tensors are allocated once at their largest sizes ("transformers continuous_batching",
setup_static_tensors).  The bench's end-to-end figure replays pa_decode the same way.  A
replay issues the captured launches with the captured arguments: the programmatic
dependent launches inside a call (the split kernel and its combine; the prefill kernel
and the single-row decode beside it) and the fused store must give the same bits as the
call issued eagerly on the same inputs, whatever the query tensor holds at replay time.
"""
import pytest
import torch

import paged_kv_attention_03_gb300 as pa
from paged_kv_attention_03_gb300.inputs import Workload, make_case_from_lengths

from _parity import assert_parity, device_tensors, host_inputs, oracle_attention

pytestmark = pytest.mark.gpu


def _capture(call):
    """Run `call` once eagerly (the library's one-time set-up happens outside the capture),
    once on a side stream, then capture it; returns the graph."""
    call()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    torch.cuda.synchronize()
    return graph


def _replay_against_eager(graph, call, q, out, cuda, rounds=3, seed=100):
    """New query contents (same address) before every replay; each replay's output must
    be the eager call's bits on the same inputs.  Returns the last replay's output."""
    got = None
    for r in range(rounds):
        gen = torch.Generator(device=cuda).manual_seed(seed + r)
        q.copy_(torch.randn(q.shape, generator=gen, device=cuda).to(torch.bfloat16))
        graph.replay()
        torch.cuda.synchronize()
        got = out.clone()
        call()
        torch.cuda.synchronize()
        assert torch.equal(got, out), f"replay {r} differs from the eager call"
    return got


@pytest.mark.parametrize("splits", [1, 3, 0])  # one split (no combine), forced, planned
def test_decode_graph_replay_matches_eager(cuda, splits):
    w = Workload("gd", 32, 8, 128, 16, ())
    case = make_case_from_lengths(w, [0, 15, 700, 2047, 3000], [1] * 5, seed=91, device=cuda)
    m = device_tensors(case, cuda)
    max_len = int(case.seq_lens.max())
    need = pa.pa_decode_workspace_size(5, 32, 8, 128, max_len, 0, splits)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=cuda)
    out = torch.empty_like(case.q)

    def call():
        pa.pa_decode(case.q, case.k_cache, case.v_cache, m["block_table"], m["seq_lens"],
                     max_len, w.final_scale, 0, splits, key=case.key, value=case.value,
                     slot_mapping=m["slot_mapping"], out=out, workspace=ws)

    graph = _capture(call)
    got = _replay_against_eager(graph, call, case.q, out, cuda)
    assert pa.pa_read_device_error(device=cuda) == 0
    # The cache already holds the stored tokens; the oracle attends the current query.
    assert_parity(got, oracle_attention(case, host_inputs(case)), "decode graph replay")


def test_mixed_prefill_graph_replay_matches_eager(cuda):
    # Prefill rows (200, 129 new tokens) and single-row sequences, which the call hands to
    # the decode launch beside the prefill kernel; the new tokens are stored by the call.
    w = Workload("gp", 32, 8, 128, 16, ())
    case = make_case_from_lengths(w, [0, 5, 300, 1000], [200, 1, 129, 1], seed=92, device=cuda)
    m = device_tensors(case, cuda)
    out = torch.empty_like(case.q)

    def call():
        pa.pa_varlen_prefill(case.q, case.k_cache, case.v_cache, m["cu_seqlens_q"],
                             m["seq_lens"], m["block_table"], case.max_query_len,
                             case.max_seq_len, w.final_scale, 0, key=case.key, value=case.value,
                             slot_mapping=m["slot_mapping"], out=out)

    graph = _capture(call)
    got = _replay_against_eager(graph, call, case.q, out, cuda, seed=200)
    assert pa.pa_read_device_error(device=cuda) == 0
    assert_parity(got, oracle_attention(case, host_inputs(case)), "varlen prefill graph replay")
