"""pa_cascade_decode against the fp64 oracle (max-abs <= 1e-2, mean-abs <= 1e-3).

"05 Attention Backends", section 8 and Q&A 4: requests sharing a cached prefix attend it
once together, their own suffixes apart, and the results are merged.  The oracle is the
plain attention over each request's whole block table (cascade is an exact
re-association of it).
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_03_gb300 as pa
from paged_kv_attention_03_gb300.inputs import Workload, make_shared_prefix_case

from _parity import assert_parity, host_inputs, oracle_attention

pytestmark = pytest.mark.gpu


def _shared_case(dev, H, Hkv, D, prefix_blocks, suffix_lens, seed, bs=16):
    """Decode requests whose first prefix_blocks blocks are the same physical blocks."""
    w = Workload("cas", H, Hkv, D, bs, ())
    return make_shared_prefix_case(w, prefix_blocks, suffix_lens, seed, dev), prefix_blocks * bs


def _cascade(case, dev, P, window=0):
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=dev)
    return pa.pa_cascade_decode(case.q, case.k_cache, case.v_cache, t(case.block_table),
                                t(case.seq_lens), int(case.seq_lens.max()), P,
                                case.workload.final_scale, window)


def _check(case, dev, P, window=0):
    out = _cascade(case, dev, P, window)
    assert pa.pa_read_device_error(device=dev) == 0
    ref = oracle_attention(case, host_inputs(case), window=window)
    return assert_parity(out, ref, f"cascade P={P} window={window}")


@pytest.mark.parametrize("window", [0, 300, 2000])
def test_cascade_matches_oracle(cuda, window):
    rng = np.random.default_rng(90)
    case, P = _shared_case(cuda, 32, 8, 128, 64, rng.integers(1, 700, size=64), seed=90)
    assert pa.pa_common_prefix_blocks(case.block_table, case.seq_lens, 16) >= 64
    _check(case, cuda, P, window)


@pytest.mark.parametrize("H,Hkv,D", [(40, 8, 128), (8, 8, 64), (64, 2, 128)])
def test_cascade_head_shapes(cuda, H, Hkv, D):
    rng = np.random.default_rng(91)
    case, P = _shared_case(cuda, H, Hkv, D, 20, rng.integers(1, 300, size=9), seed=91)
    _check(case, cuda, P)


@pytest.mark.parametrize("batch", [1, 300])
def test_cascade_batch_sizes(cuda, batch):
    # 300 requests with G = 4 need three query-tile pairs per kv head.
    rng = np.random.default_rng(92)
    case, P = _shared_case(cuda, 32, 8, 128, 33, rng.integers(1, 200, size=batch), seed=92)
    _check(case, cuda, P)


def test_cascade_prefix_zero_and_prefix_only_requests(cuda):
    rng = np.random.default_rng(93)
    case, P = _shared_case(cuda, 32, 8, 128, 8, rng.integers(1, 100, size=5), seed=93)
    _check(case, cuda, 0)  # no shared part: plain decode through the same path
    # A request whose every key is in the prefix (its suffix part is empty).
    case2, P2 = _shared_case(cuda, 32, 8, 128, 8, [0, 40, 3], seed=94)
    _check(case2, cuda, P2)


def test_cascade_long_prefix_short_suffixes(cuda):
    # An 8192-key shared prefix and suffixes of 1..8 keys: the suffix decode runs beside
    # the prefix kernel and finishes first, so the merge must still wait for the prefix.
    rng = np.random.default_rng(95)
    case, P = _shared_case(cuda, 32, 8, 128, 512, rng.integers(1, 9, size=32), seed=95)
    _check(case, cuda, P)
