"""CPU-side checks of the C ABI: the library loads, exports every declared entry point,
and rejects invalid arguments on the host before launching anything."""
import ctypes
import os
import re

import pytest

import paged_kv_attention_03_gb300 as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa_gb300.h")

OK, INVALID, UNSUPPORTED = pa.PA_OK, pa.PA_ERR_INVALID_ARG, pa.PA_ERR_UNSUPPORTED
FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced on these paths
MISALIGNED = 0x10002


@pytest.fixture(scope="module")
def lib():
    pa.build()
    return pa.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert names == sorted(pa.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    assert "sm_103a" in pa.version()
    assert pa.status_string(0) == "PA_OK"
    assert pa.status_string(4) == "PA_ERR_DEVICE_CHECK"


def _decode(lib, **kw):
    a = dict(out=FAKE, q=FAKE, key=None, value=None, slot=None, kc=FAKE, vc=FAKE, bt=FAKE,
             max_blocks=8, seq_lens=FAKE, batch=2, max_seq_len=100, num_blocks=16, bs=16,
             H=8, Hkv=2, D=128, window=0, scale=0.1, splits=1, ws=None, ws_bytes=0)
    a.update(kw)
    return lib.pa_decode(a["out"], a["q"], a["key"], a["value"], a["slot"], a["kc"], a["vc"],
                         a["bt"], a["max_blocks"], a["seq_lens"], a["batch"], a["max_seq_len"],
                         a["num_blocks"], a["bs"], a["H"], a["Hkv"], a["D"], a["window"],
                         a["scale"], a["splits"], a["ws"], a["ws_bytes"], None)


def _prefill(lib, **kw):
    a = dict(out=FAKE, q=FAKE, key=None, value=None, slot=None, kc=FAKE, vc=FAKE, cuq=FAKE,
             cuk=None, seq_lens=FAKE, bt=FAKE, max_blocks=8, num_seqs=2, total_q=10, mq=8,
             mk=100, num_blocks=16, bs=16, H=8, Hkv=2, D=128, window=0, scale=0.1)
    a.update(kw)
    return lib.pa_varlen_prefill(a["out"], a["q"], a["key"], a["value"], a["slot"], a["kc"],
                                 a["vc"], a["cuq"], a["cuk"], a["seq_lens"], a["bt"],
                                 a["max_blocks"], a["num_seqs"], a["total_q"], a["mq"], a["mk"],
                                 a["num_blocks"], a["bs"], a["H"], a["Hkv"], a["D"],
                                 a["window"], a["scale"], None)


def test_store_argument_checks(lib):
    s = lib.pa_store_kvcache
    assert s(None, None, None, None, None, 0, 4, 16, 2, 64, None) == OK  # nothing to do
    assert s(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 4, 16, 2, 64, None) == INVALID
    assert s(None, FAKE, FAKE, FAKE, FAKE, 3, 4, 16, 2, 64, None) == INVALID
    assert s(FAKE, FAKE, FAKE, FAKE, FAKE, 3, 4, 0, 2, 64, None) == INVALID
    assert s(FAKE, FAKE, FAKE, FAKE, FAKE, 3, 4, 16, 1, 4, None) == UNSUPPORTED  # row not 16 B
    assert s(MISALIGNED, FAKE, FAKE, FAKE, FAKE, 3, 4, 16, 2, 64, None) == INVALID


def test_decode_argument_checks(lib):
    assert _decode(lib, batch=0) == OK
    assert _decode(lib, D=96) == UNSUPPORTED  # head sizes built: 64, 128
    assert _decode(lib, H=6, Hkv=4) == INVALID  # num_heads % num_kv_heads != 0
    assert _decode(lib, bs=24) == UNSUPPORTED  # block_size must be a power of two
    assert _decode(lib, H=130, Hkv=2) == UNSUPPORTED  # group of 65 > 64
    assert _decode(lib, key=FAKE) == INVALID  # key without value / slot_mapping
    assert _decode(lib, q=None) == INVALID
    assert _decode(lib, q=MISALIGNED) == INVALID
    assert _decode(lib, max_seq_len=-1) == INVALID
    # splits > 1 need a workspace of the advertised size
    assert _decode(lib, splits=4, ws=None, ws_bytes=0, max_seq_len=4096) == INVALID
    need = pa.pa_decode_workspace_size(2, 8, 2, 128, 4096, 0, 4)
    assert need > 0
    assert _decode(lib, splits=4, ws=FAKE, ws_bytes=need - 1, max_seq_len=4096) == INVALID
    assert _decode(lib, splits=4, ws=FAKE + 16, ws_bytes=need, max_seq_len=4096) == INVALID


def test_prefill_argument_checks(lib):
    assert _prefill(lib, num_seqs=0) == OK
    assert _prefill(lib, total_q=0) == OK
    assert _prefill(lib, D=256) == UNSUPPORTED
    assert _prefill(lib, bs=8) == UNSUPPORTED  # prefill pages are at least 16 rows
    assert _prefill(lib, H=10, Hkv=4) == INVALID
    assert _prefill(lib, mq=200, mk=100) == INVALID  # more queries than keys
    assert _prefill(lib, seq_lens=None, cuk=None) == INVALID
    assert _prefill(lib, cuq=None) == INVALID
    assert _prefill(lib, slot=FAKE) == INVALID
    assert _prefill(lib, out=MISALIGNED) == INVALID
    assert _prefill(lib, scale=0.0) == INVALID
    assert _prefill(lib, scale=-0.1) == INVALID


def test_decode_split_plan_is_consistent(lib):
    for batch, H, Hkv, L, w, req in [(64, 32, 8, 4096, 0, 0), (8, 40, 8, 131072, 0, 0),
                                     (4, 8, 2, 100, 0, 0), (128, 32, 8, 8704, 4096, 0),
                                     (3, 8, 8, 5000, 0, 7), (1, 8, 1, 16, 0, 3)]:
        n = pa.pa_decode_num_splits(batch, H, Hkv, 128, L, w, req)
        assert n >= 1
        if req:
            assert n <= req
        ws = pa.pa_decode_workspace_size(batch, H, Hkv, 128, L, w, req)
        assert (ws == 0) == (n == 1)
        if n > 1:
            assert ws >= batch * H * n * (128 + 2) * 4
    assert pa.pa_decode_num_splits(1, 6, 4, 128, 10, 0, 0) == 0  # invalid -> 0


def test_read_device_error_without_gpu_reports_cuda_error(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("only meaningful on a machine without a GPU")
    flags = ctypes.c_uint32(0)
    assert lib.pa_read_device_error(None, ctypes.byref(flags), 0) == pa.PA_ERR_CUDA
    # The CUDA error behind that status is kept for the calling thread.
    text = lib.pa_last_cuda_error_string().decode()
    assert text and text != "no error"
    with pytest.raises(pa.PAError, match=r"PA_ERR_CUDA \(.+\)"):
        raise pa.PAError(pa.PA_ERR_CUDA, "probe")


def test_common_prefix_blocks_matches_brute_force():
    import numpy as np
    rng = np.random.default_rng(5)
    for trial in range(200):
        batch = int(rng.integers(1, 6))
        mb = int(rng.integers(1, 9))
        bs = 16
        base = rng.integers(0, 50, size=mb)
        bt = np.tile(base, (batch, 1)).astype(np.int32)
        for b in range(1, batch):  # each row diverges somewhere (or never)
            k = int(rng.integers(0, mb + 1))
            if k < mb:
                bt[b, k:] = rng.integers(50, 100, size=mb - k)
        sl = rng.integers(0, mb * bs + 1, size=batch).astype(np.int32)
        want = 0
        while (want < mb and all(bt[b, want] == bt[0, want] for b in range(batch))
               and all((want + 1) * bs <= sl[b] for b in range(batch))):
            want += 1
        assert pa.pa_common_prefix_blocks(bt, sl, bs) == want, (bt, sl)


def test_cascade_argument_checks(lib):
    # prefix_len must be a multiple of block_size and within max_seq_len (host checks).
    p = ctypes.c_void_p(16)
    bad = lib.pa_cascade_decode(p, p, p, p, p, 4, p, 2, 100, 17, 10, 16, 8, 2, 128, 0,
                                ctypes.c_float(0.1), p, 1 << 20, None)
    assert bad == pa.PA_ERR_INVALID_ARG
    bad = lib.pa_cascade_decode(p, p, p, p, p, 4, p, 2, 100, 112, 10, 16, 8, 2, 128, 0,
                                ctypes.c_float(0.1), p, 1 << 20, None)
    assert bad == pa.PA_ERR_INVALID_ARG
    assert lib.pa_cascade_decode(p, p, p, p, p, 4, p, 2, 100, 16, 10, 8, 8, 2, 128, 0,
                                 ctypes.c_float(0.1), p, 1 << 20, None) == pa.PA_ERR_UNSUPPORTED
