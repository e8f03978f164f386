"""pa_decode_noalloc: the decode entry point for callers that cannot allocate device
memory (its split-K scratch is a fixed array inside the library).

Checked through the C ABI against pa_decode, which runs the same kernels with the same
split plan on a caller-provided workspace: the outputs must be bit-identical, on two
calls in a row with different shapes and split counts (a stale or misplaced partial
from the shared scratch would change bits).  The first case is also checked against
the oracle within the attention tolerance.  This file is collected last.
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_03_gb300 as pa
from paged_kv_attention_03_gb300.inputs import make_case

from _parity import assert_parity, host_inputs, oracle_attention

pytestmark = pytest.mark.gpu


def _args(case, dev, num_splits):
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=dev)
    w = case.workload
    return dict(q=case.q, k_cache=case.k_cache, v_cache=case.v_cache,
                block_table=t(case.block_table), seq_lens=t(case.seq_lens),
                max_seq_len=case.max_seq_len, scale=w.final_scale,
                sliding_window=w.sliding_window, num_splits=num_splits)


def test_noalloc_decode_matches_workspace_decode_twice(cuda):
    cases = [(make_case("long_decode_small", seed=51, device=cuda), 0),
             (make_case("batched_decode_small", seed=52, device=cuda), 3)]
    for case, splits in cases:
        w = case.workload
        assert pa.pa_decode_num_splits(case.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                       case.max_seq_len, w.sliding_window, splits) > 1
    for i, (case, splits) in enumerate(cases):  # two calls in a row
        a = _args(case, cuda, splits)
        ref = pa.pa_decode(**a)
        out = torch.full_like(case.q, float("nan"))
        pa.pa_decode_noalloc(**a, out=out)
        assert pa.pa_read_device_error(device=cuda) == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), \
            f"call {i}: output differs from pa_decode"
        if i == 0:
            assert_parity(out, oracle_attention(case, host_inputs(case)), "noalloc vs oracle")


def test_noalloc_decode_rejects_scratch_beyond_its_limit(cuda):
    case = make_case("batched_decode_small", seed=53, device=cuda)
    a = _args(case, cuda, 1024)
    a["max_seq_len"] = 1 << 20  # needs far more than the fixed scratch
    need = pa.pa_decode_workspace_size(case.num_seqs, 32, 8, 128, 1 << 20, 0, 1024)
    assert need > (16 << 20)
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_noalloc(**a)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
