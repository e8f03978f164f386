"""Plain fp64 CPU oracle for attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library never
imports, links or calls it, and it imports nothing from the CUDA package: the two
sides meet only in the tests, on the same seeded inputs.

The arithmetic lives in ``pa_oracle.c`` (plain C, fp64, one pthread pool); this
module compiles it with the host C compiler on first use and wraps it with ctypes.
Arrays are numpy: bf16 tensors travel as their uint16 bit patterns, indices as
int32, results come back as float64.

Functions and the passages they follow (page title and section):

* :func:`store_kvcache` -- "MinivLLM API docs - Attention", store_kvcache: slot s
  goes to block s // block_size, row s % block_size; slot -1 (any negative) skips.
* :func:`mask` -- "transformers continuous_batching/input_ouputs.py",
  build_attention_mask: bottom-right causal alignment plus a window of w keys
  that includes the query's own position.
* :func:`paged_attention` / :func:`attend_row` -- the gather through block_tables
  ("MinivLLM API docs - Attention", paged_attention_decode), GQA head mapping
  h -> h // (num_heads / num_kv_heads) ("vllm-npu 0.4.2, torch_sdpa.py"), and
  o = softmax(scale * q K^T) V over the visible keys, all in fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "libpa_oracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, ERANGE, ENOMEM = 0, -1, -2, -3


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into libpa_oracle.so next to it (plain gcc, no GPU)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    cc = os.environ.get("CC", "gcc")
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        p = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.pa_oracle_store_kvcache.argtypes = [p, p, p, p, p, i64, i64, i32, i32, i32]
        lib.pa_oracle_store_kvcache.restype = i32
        lib.pa_oracle_mask.argtypes = [i32, i32, i32, p]
        lib.pa_oracle_mask.restype = i32
        lib.pa_oracle_attend_row.argtypes = [p, p, p, p, p, i64, i64, i32, i32, i32, i32,
                                             i64, i32, dbl, p]
        lib.pa_oracle_attend_row.restype = i32
        lib.pa_oracle_attend_row_state.argtypes = [p, p, p, p, p, p, i64, i64, i64, i32, i32,
                                                   i32, i32, i64, i32, dbl, p]
        lib.pa_oracle_attend_row_state.restype = i32
        lib.pa_oracle_merge_states.argtypes = [p, p, p, p, i32, i64, i32]
        lib.pa_oracle_merge_states.restype = i32
        lib.pa_oracle_fp8_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.pa_oracle_fp8_e4m3_decode.restype = dbl
        lib.pa_oracle_fp8_e4m3_encode.argtypes = [ctypes.c_float]
        lib.pa_oracle_fp8_e4m3_encode.restype = ctypes.c_uint8
        lib.pa_oracle_store_kvcache_fp8.argtypes = [p, p, p, p, p, i64, i64, i32, i32, i32,
                                                    ctypes.c_float]
        lib.pa_oracle_store_kvcache_fp8.restype = i32
        lib.pa_oracle_paged_attention_fp8.argtypes = [p, p, p, p, p, p, p, i64, i32, i32, i32,
                                                      i32, i32, i64, i32, dbl, dbl, i32]
        lib.pa_oracle_paged_attention_fp8.restype = i32
        lib.pa_oracle_paged_attention.argtypes = [p, p, p, p, p, p, p, i64, i32, i32, i32,
                                                  i32, i32, i64, i32, dbl, i32]
        lib.pa_oracle_paged_attention.restype = i32
        lib.pa_oracle_default_threads.argtypes = []
        lib.pa_oracle_default_threads.restype = i32
        lib.pa_oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.pa_oracle_bf16_to_double.restype = dbl
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 data must be passed as uint16 bit patterns, got {a.dtype}")
    return a


def _i32(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.int32:
        raise TypeError(f"index arrays must be int32, got {a.dtype}")
    return a


def _check(rc: int, what: str) -> None:
    if rc != OK:
        name = {EINVAL: "invalid argument", ERANGE: "block index out of range",
                ENOMEM: "out of memory"}.get(rc, str(rc))
        raise OracleError(f"oracle {what}: {name}")


def default_threads() -> int:
    return int(_load().pa_oracle_default_threads())


def bf16_to_double(bits: int) -> float:
    return float(_load().pa_oracle_bf16_to_double(int(bits) & 0xFFFF))


def store_kvcache(key, value, k_cache, v_cache, slot_mapping, block_size: int) -> None:
    """In place: k_cache/v_cache [num_blocks, block_size, num_kv_heads, head_dim] uint16.

    key/value [num_tokens, num_kv_heads, head_dim] uint16; slot_mapping [num_tokens]
    int32.
    """
    lib = _load()
    key, value = _u16(key), _u16(value)
    if not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
        raise ValueError("caches must be C-contiguous")
    kc, vc = _u16(k_cache), _u16(v_cache)
    slots = _i32(slot_mapping)
    nb, bs, hkv, d = kc.shape
    if bs != block_size:
        raise ValueError("block_size does not match the cache shape")
    rc = lib.pa_oracle_store_kvcache(_ptr(key), _ptr(value), _ptr(kc), _ptr(vc),
                                     _ptr(slots), slots.shape[0], nb, bs, hkv, d)
    _check(rc, "store_kvcache")


def mask(sq: int, sk: int, window: int) -> np.ndarray:
    """[sq, sk] bool: which keys each of the sq newest queries may attend to."""
    out = np.zeros((max(sq, 0), max(sk, 0)), dtype=np.uint8)
    rc = _load().pa_oracle_mask(sq, sk, window, _ptr(out))
    _check(rc, "mask")
    return out.astype(bool)


def attend_row(q_row, k_cache, v_cache, block_table_row, seq_len: int, pos: int,
               num_heads: int, num_kv_heads: int, window: int, scale: float) -> np.ndarray:
    """One query row (all heads) at absolute position ``pos``; returns [H, D] float64."""
    lib = _load()
    q_row, kc, vc = _u16(q_row), _u16(k_cache), _u16(v_cache)
    bt = _i32(block_table_row)
    nb, bs, hkv, d = kc.shape
    out = np.zeros((num_heads, d), dtype=np.float64)
    rc = lib.pa_oracle_attend_row(_ptr(out), _ptr(q_row), _ptr(kc), _ptr(vc), _ptr(bt),
                                  int(seq_len), int(pos), num_heads, num_kv_heads, d, bs,
                                  nb, int(window), float(scale), None)
    _check(rc, "attend_row")
    return out


def attend_row_state(q_row, k_cache, v_cache, block_table_row, seq_len: int, pos: int,
                     key_begin: int, num_heads: int, num_kv_heads: int, window: int,
                     scale: float) -> tuple[np.ndarray, np.ndarray]:
    """Partial result of one query row over its visible keys j >= key_begin: the row
    [H, D] and lse [H] (natural log; -inf with a zero row when no key is left)."""
    lib = _load()
    q_row, kc, vc = _u16(q_row), _u16(k_cache), _u16(v_cache)
    bt = _i32(block_table_row)
    nb, bs, hkv, d = kc.shape
    out = np.zeros((num_heads, d), dtype=np.float64)
    lse = np.zeros(num_heads, dtype=np.float64)
    rc = lib.pa_oracle_attend_row_state(_ptr(out), _ptr(lse), _ptr(q_row), _ptr(kc), _ptr(vc),
                                        _ptr(bt), int(seq_len), int(pos), int(key_begin),
                                        num_heads, num_kv_heads, d, bs, nb, int(window),
                                        float(scale), None)
    _check(rc, "attend_row_state")
    return out, lse


def fp8_e4m3_decode(code: int) -> float:
    """Value of one FP8 E4M3 code (NaN for S.1111.111)."""
    return float(_load().pa_oracle_fp8_e4m3_decode(int(code) & 0xFF))


def fp8_e4m3_encode(x: float) -> int:
    """Nearest E4M3 code to the fp32 value x (ties to even, saturating at 448)."""
    return int(_load().pa_oracle_fp8_e4m3_encode(float(np.float32(x))))


def store_kvcache_fp8(key, value, k_cache, v_cache, slot_mapping, block_size: int,
                      kv_scale: float) -> None:
    """store_kvcache into FP8 E4M3 caches (uint8 [NB, bs, Hkv, D], in place):
    code = encode(x / kv_scale) with x the bf16 input and the division in fp32."""
    lib = _load()
    key, value = _u16(key), _u16(value)
    if k_cache.dtype != np.uint8 or v_cache.dtype != np.uint8:
        raise TypeError("fp8 caches are uint8 arrays")
    sm = _i32(slot_mapping)
    t = key.shape[0]
    nb, bs, hkv, d = k_cache.shape
    _check(lib.pa_oracle_store_kvcache_fp8(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                           _ptr(sm), t, nb, bs, hkv, d, float(kv_scale)),
           "store_kvcache_fp8")


def paged_attention_fp8(q, k_cache, v_cache, cu_seqlens_q, seq_lens, block_table,
                        num_heads: int, num_kv_heads: int, window: int, scale: float,
                        kv_scale: float, num_threads: int = 0) -> np.ndarray:
    """paged_attention over FP8 E4M3 caches (uint8) whose elements read code * kv_scale."""
    lib = _load()
    q = _u16(q)
    if k_cache.dtype != np.uint8 or v_cache.dtype != np.uint8:
        raise TypeError("fp8 caches are uint8 arrays")
    kc, vc = np.ascontiguousarray(k_cache), np.ascontiguousarray(v_cache)
    cu, sl, bt = _i32(cu_seqlens_q), _i32(seq_lens), _i32(block_table)
    nb, bs, hkv, d = kc.shape
    out = np.zeros((q.shape[0], num_heads, d), dtype=np.float64)
    _check(lib.pa_oracle_paged_attention_fp8(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(cu),
                                             _ptr(sl), _ptr(bt), bt.shape[1], len(sl),
                                             num_heads, num_kv_heads, d, bs, nb, int(window),
                                             float(scale), float(kv_scale), num_threads),
           "paged_attention_fp8")
    return out


def merge_states(states, lses) -> tuple[np.ndarray, np.ndarray]:
    """Merge R partial results: states [R, rows, D], lses [R, rows] (float64).
    Returns (out [rows, D], lse [rows])."""
    lib = _load()
    st = np.ascontiguousarray(states, dtype=np.float64)
    ls = np.ascontiguousarray(lses, dtype=np.float64)
    r, rows, d = st.shape
    if ls.shape != (r, rows):
        raise ValueError("lses must be [R, rows]")
    out = np.zeros((rows, d), dtype=np.float64)
    lse = np.zeros(rows, dtype=np.float64)
    _check(lib.pa_oracle_merge_states(_ptr(out), _ptr(lse), _ptr(st), _ptr(ls), r, rows, d),
           "merge_states")
    return out, lse


def paged_attention(q, k_cache, v_cache, cu_seqlens_q, seq_lens, block_table,
                    num_heads: int, num_kv_heads: int, window: int, scale: float,
                    num_threads: int = 0) -> np.ndarray:
    """Packed varlen (or decode, with cu_seqlens_q = 0..B) paged attention in fp64.

    q: [total_q, num_heads, head_dim] uint16; caches [NB, bs, Hkv, D] uint16;
    cu_seqlens_q [num_seqs + 1], seq_lens [num_seqs], block_table [num_seqs, max_blocks]
    int32.  Returns [total_q, num_heads, head_dim] float64.
    """
    lib = _load()
    q, kc, vc = _u16(q), _u16(k_cache), _u16(v_cache)
    cu, sl, bt = _i32(cu_seqlens_q), _i32(seq_lens), _i32(block_table)
    nb, bs, hkv, d = kc.shape
    if hkv != num_kv_heads:
        raise ValueError("num_kv_heads does not match the cache shape")
    num_seqs = sl.shape[0]
    if bt.ndim != 2 or bt.shape[0] != num_seqs or cu.shape[0] != num_seqs + 1:
        raise ValueError("block_table / cu_seqlens_q shapes do not match seq_lens")
    out = np.zeros((q.shape[0], num_heads, d), dtype=np.float64)
    rc = lib.pa_oracle_paged_attention(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(cu),
                                       _ptr(sl), _ptr(bt), bt.shape[1], num_seqs,
                                       num_heads, num_kv_heads, d, bs, nb, int(window),
                                       float(scale), int(num_threads))
    _check(rc, "paged_attention")
    return out
