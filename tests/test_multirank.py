"""Host-side multi-rank logic of bench.py, on CPU with the gloo backend (world size 2).

The path shards with no data exchange (each rank runs its own replica), so what is
tested is the plumbing around it: rank discovery, distinct per-rank inputs, the
max-over-ranks timing and the sum-over-ranks work count that make `value`.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_attention_03_gb300.inputs import make_case

    r, local, ws = bench._dist()
    assert (r, local, ws) == (rank, rank, world)
    case = make_case("tiny_decode", seed=r)  # one replica per rank, own seed
    t = bench._max_over_ranks(1.0 + r, ws, "cpu")
    n = bench._sum_over_ranks(float(bench.decode_kv_bytes(case)), ws, "cpu")
    bench._barrier(ws)
    q.put((r, t, n, case.q.float().sum().item()))
    torch.distributed.destroy_process_group()


def test_two_rank_timing_and_work_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, t0, n0, s0), (r1, t1, n1, s1) = res
    assert t0 == t1 == 2.0  # max over ranks of 1.0 and 2.0
    assert n0 == n1 and n0 > 0  # both ranks see the total work
    assert s0 != s1  # distinct per-rank inputs


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny_decode", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["unit"] == "GB/s"
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0


def _dcp_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    from paged_kv_attention_03_gb300.dcp import gather_states

    g = torch.Generator().manual_seed(100 + rank)
    state = torch.randn(3, 4, 8, generator=g)        # [batch, heads, head_dim]
    lse = torch.randn(3, 4, generator=g) * 5
    if rank == 1:
        lse[0, 0] = float("-inf")                    # this rank has no key for one row
    states, lses = gather_states(state, lse)
    q.put((rank, state.numpy(), lse.numpy(), states.numpy(), lses.numpy()))
    torch.distributed.destroy_process_group()


def test_context_parallel_exchange_two_ranks():
    # The exchange step of context-parallel decode: every rank ends with all ranks'
    # partial results in rank order; merging them is the merge of their key sets.
    import numpy as np
    import oracle

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dcp_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=120) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    own_states = np.stack([r[1] for r in res])
    own_lses = np.stack([r[2] for r in res])
    for _, _, _, states, lses in res:
        np.testing.assert_array_equal(states, own_states)
        np.testing.assert_array_equal(lses, own_lses)
    # Row (0, 0) has keys only on rank 0: the merge must return rank 0's row there.
    merged, merged_lse = oracle.merge_states(own_states.reshape(2, -1, 8).astype(np.float64),
                                             own_lses.reshape(2, -1).astype(np.float64))
    np.testing.assert_allclose(merged[0], own_states[0, 0, 0], rtol=0, atol=1e-6)
    assert merged_lse[0] == pytest.approx(float(own_lses[0, 0, 0]), abs=1e-6)


@pytest.mark.parametrize("interleave", [0, 1, 16, 64])
def test_dcp_key_begin_counts_the_keys_before_the_window(interleave):
    # CPU: each rank's first visible local key is the number of its keys whose global
    # position lies before the window (brute force over the deal).
    import numpy as np
    import torch
    from paged_kv_attention_03_gb300.dcp import dcp_key_begin

    rng = np.random.default_rng(5)
    lens = rng.integers(1, 5000, size=40).astype(np.int32)
    world = 3
    for window in (1, 7, 100, 4999, 6000):
        for r in range(world):
            if interleave:
                owned = [np.nonzero((np.arange(L) // interleave) % world == r)[0] for L in lens]
                starts = None
            else:
                st = (lens.astype(np.int64) * r) // world
                en = (lens.astype(np.int64) * (r + 1)) // world
                owned = [np.arange(a, b) for a, b in zip(st, en)]
                starts = torch.as_tensor(st.astype(np.int32))
            nloc = torch.as_tensor(np.array([len(o) for o in owned], dtype=np.int32))
            kb = dcp_key_begin(torch.as_tensor(lens), window, r, world, interleave, starts, nloc)
            want = [int(np.sum(o < max(0, int(L) - window))) for o, L in zip(owned, lens)]
            assert kb.tolist() == want, (interleave, window, r)
