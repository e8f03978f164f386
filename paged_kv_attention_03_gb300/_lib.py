"""ctypes binding of libpa_gb300.so (the C ABI declared in include/pa_gb300.h).

Argument marshalling only: tensors become raw device pointers, the current CUDA
stream becomes a cudaStream_t, and every computation runs in the library's kernels.
There is no CPU path: if the library is missing or a call fails, an exception says
so.
"""
from __future__ import annotations

import contextlib
import ctypes
import functools
import os
import threading

import torch

from . import builder as _build

_lock = threading.Lock()
_lib = None

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_DEVICE_CHECK = range(5)
DEVERR_SLOT_RANGE = 0x1
DEVERR_BLOCK_RANGE = 0x2
DEVERR_SEQ_RANGE = 0x4
DEVERR_QUERY_LEN = 0x8
DEVERR_SEQLENS_K = 0x10
DEVERR_TIMEOUT = 0x20
DEVERR_SLOT_MISMATCH = 0x40

EXPORTED = ("pa_status_string", "pa_version", "pa_store_kvcache", "pa_decode_num_splits",
            "pa_decode_workspace_size", "pa_decode", "pa_varlen_prefill",
            "pa_read_device_error", "pa_decode_noalloc", "pa_last_cuda_error_string",
            "pa_decode_state_workspace_size", "pa_decode_state", "pa_merge_states",
            "pa_cascade_decode_workspace_size", "pa_cascade_decode", "pa_common_prefix_blocks",
            "pa_store_kvcache_fp8", "pa_decode_fp8", "pa_debug_prefill_stall",
            "pa_varlen_prefill_fp8")


class PAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {status_string(status)}"
        if status == PA_ERR_CUDA:
            msg += f" ({last_cuda_error_string()})"
        super().__init__(msg)


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load the shared library (building it first if it is missing and allowed)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"libpa_gb300.so is not built ({path}); run build()")
            _build.build()
        lib = ctypes.CDLL(path)
        vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                 ctypes.c_float, ctypes.c_size_t)
        lib.pa_status_string.argtypes = [ctypes.c_int]
        lib.pa_status_string.restype = ctypes.c_char_p
        lib.pa_version.argtypes = []
        lib.pa_version.restype = ctypes.c_char_p
        lib.pa_last_cuda_error_string.argtypes = []
        lib.pa_last_cuda_error_string.restype = ctypes.c_char_p
        lib.pa_store_kvcache.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, i32, i32, vp]
        lib.pa_store_kvcache.restype = ctypes.c_int
        lib.pa_decode_num_splits.argtypes = [i32] * 7
        lib.pa_decode_num_splits.restype = ctypes.c_int
        lib.pa_decode_workspace_size.argtypes = [i32] * 7
        lib.pa_decode_workspace_size.restype = sz
        lib.pa_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i64, i32,
                                  i32, i32, i32, i32, f32, i32, vp, sz, vp]
        lib.pa_decode.restype = ctypes.c_int
        lib.pa_varlen_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                          i32, i32, i32, i64, i32, i32, i32, i32, i32, f32, vp]
        lib.pa_varlen_prefill.restype = ctypes.c_int
        lib.pa_decode_state_workspace_size.argtypes = [i32] * 7
        lib.pa_decode_state_workspace_size.restype = sz
        lib.pa_decode_state.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i64, i32,
                                        i32, i32, i32, i32, f32, i32, vp, sz, vp]
        lib.pa_decode_state.restype = ctypes.c_int
        lib.pa_merge_states.argtypes = [vp, vp, vp, vp, vp, i32, i64, i32, vp]
        lib.pa_merge_states.restype = ctypes.c_int
        lib.pa_cascade_decode_workspace_size.argtypes = [i32] * 7
        lib.pa_cascade_decode_workspace_size.restype = sz
        lib.pa_cascade_decode.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i64, i32,
                                          i32, i32, i32, i32, f32, vp, sz, vp]
        lib.pa_cascade_decode.restype = ctypes.c_int
        lib.pa_common_prefix_blocks.argtypes = [vp, i32, i32, vp, i32]
        lib.pa_common_prefix_blocks.restype = ctypes.c_int
        lib.pa_store_kvcache_fp8.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, i32, i32, f32,
                                             vp]
        lib.pa_store_kvcache_fp8.restype = ctypes.c_int
        lib.pa_decode_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i64,
                                      i32, i32, i32, i32, i32, f32, f32, i32, vp, sz, vp]
        lib.pa_decode_fp8.restype = ctypes.c_int
        lib.pa_read_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
        lib.pa_read_device_error.restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load().pa_status_string(int(status)).decode()
    except Exception:  # library not loadable: still describe the code
        return str(status)


def version() -> str:
    return load().pa_version().decode()


def last_cuda_error_string() -> str:
    """CUDA error text behind the most recent PA_ERR_CUDA on this thread."""
    return load().pa_last_cuda_error_string().decode()


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PAError(status, what)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return t.data_ptr()


# The current stream's raw handle without building a Stream object (about 2 us less per
# call); torch.cuda.current_stream is the fallback.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(device: torch.device) -> int:
    if _raw_stream is not None:
        idx = device.index if device.index is not None else torch.cuda.current_device()
        return _raw_stream(idx)
    return torch.cuda.current_stream(device).cuda_stream


def _need(t: torch.Tensor, dtype: torch.dtype, name: str, device: torch.device | None = None):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _out(out: torch.Tensor | None, shape, dtype: torch.dtype, dev: torch.device,
         name: str = "out") -> torch.Tensor:
    """A caller-supplied output must match exactly (the kernels write shape's bytes);
    None allocates one."""
    if out is None:
        return torch.empty(tuple(shape), dtype=dtype, device=dev)
    _need(out, dtype, name, dev)
    if tuple(out.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(out.shape)}")
    if not out.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return out


def _new_tokens(key, value, slot_mapping, rows: int, hkv: int, head_dim: int,
                dev: torch.device, what: str) -> None:
    """The optional store of new tokens: key/value [rows, Hkv, D] bf16 and slot_mapping
    [rows] int32, all three or none."""
    given = [t is not None for t in (key, value, slot_mapping)]
    if not any(given):
        return
    if not all(given):
        raise ValueError(f"{what}: key, value and slot_mapping are given together")
    _need(key, torch.bfloat16, "key", dev)
    _need(value, torch.bfloat16, "value", dev)
    _need(slot_mapping, torch.int32, "slot_mapping", dev)
    if tuple(key.shape) != (rows, hkv, head_dim) or value.shape != key.shape:
        raise ValueError(f"{what}: key/value must be [{rows}, {hkv}, {head_dim}]")
    if tuple(slot_mapping.shape) != (rows,):
        raise ValueError(f"{what}: slot_mapping must have {rows} entries")


def _on(dev: torch.device):
    """Make `dev` the current device for the call: the library takes the device of its
    error word, scratch and shared-memory limits from the current device."""
    if dev.index is None or dev.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(dev)


def pa_store_kvcache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                     v_cache: torch.Tensor, slot_mapping: torch.Tensor) -> None:
    """Scatter key/value [T, Hkv, D] into k_cache/v_cache [NB, bs, Hkv, D] by slot_mapping [T]."""
    lib = load()
    dev = k_cache.device
    for t, n in ((key, "key"), (value, "value"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n, dev)
    _need(slot_mapping, torch.int32, "slot_mapping", dev)
    nb, bs, hkv, d = k_cache.shape
    if v_cache.shape != k_cache.shape or key.shape != value.shape or key.shape[1:] != (hkv, d):
        raise ValueError("store_kvcache: inconsistent shapes")
    if slot_mapping.shape[0] != key.shape[0]:
        raise ValueError("store_kvcache: slot_mapping length != number of tokens")
    with _on(dev):
        st = lib.pa_store_kvcache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(slot_mapping), key.shape[0], nb, bs, hkv, d, _stream(dev))
    _check(st, "pa_store_kvcache")


def pa_store_kvcache_fp8(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                         v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                         kv_scale: float) -> None:
    """Store key/value [T, Hkv, D] bf16 into FP8 E4M3 caches (uint8 [NB, bs, Hkv, D]) as
    codes of x / kv_scale."""
    lib = load()
    dev = k_cache.device
    _need(key, torch.bfloat16, "key", dev)
    _need(value, torch.bfloat16, "value", dev)
    _need(k_cache, torch.uint8, "k_cache", dev)
    _need(v_cache, torch.uint8, "v_cache", dev)
    _need(slot_mapping, torch.int32, "slot_mapping", dev)
    nb, bs, hkv, d = k_cache.shape
    if v_cache.shape != k_cache.shape or key.shape != value.shape or key.shape[1:] != (hkv, d):
        raise ValueError("store_kvcache_fp8: inconsistent shapes")
    if slot_mapping.shape[0] != key.shape[0]:
        raise ValueError("store_kvcache_fp8: slot_mapping length != number of tokens")
    with _on(dev):
        st = lib.pa_store_kvcache_fp8(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(slot_mapping), key.shape[0], nb, bs, hkv, d,
                                      float(kv_scale), _stream(dev))
    _check(st, "pa_store_kvcache_fp8")


def pa_decode_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                  block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                  scale: float, kv_scale: float, sliding_window: int = 0, num_splits: int = 0,
                  key: torch.Tensor | None = None, value: torch.Tensor | None = None,
                  slot_mapping: torch.Tensor | None = None, out: torch.Tensor | None = None,
                  workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Paged decode over FP8 E4M3 caches (uint8 [NB, bs, Hkv, D], read as code * kv_scale);
    q / key / value / out bf16.  New tokens, when given, are stored in the same launch."""
    lib = load()
    dev = q.device
    _need(q, torch.bfloat16, "q", dev)
    _need(k_cache, torch.uint8, "k_cache", dev)
    _need(v_cache, torch.uint8, "v_cache", dev)
    _need(block_table, torch.int32, "block_table", dev)
    _need(seq_lens, torch.int32, "seq_lens", dev)
    batch, num_heads, head_dim = q.shape
    nb, bs, hkv, d = k_cache.shape
    if d != head_dim or block_table.dim() != 2 or block_table.shape[0] != batch:
        raise ValueError("pa_decode_fp8: inconsistent shapes")
    _new_tokens(key, value, slot_mapping, batch, hkv, head_dim, dev, "pa_decode_fp8")
    out = _out(out, q.shape, torch.bfloat16, dev)
    need = pa_decode_workspace_size(batch, num_heads, hkv, head_dim, max_seq_len,
                                    sliding_window, num_splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = _ptr(workspace) if need else None
    ws_bytes = workspace.numel() * workspace.element_size() if need else 0
    with _on(dev):
        st = lib.pa_decode_fp8(_ptr(out), _ptr(q), _ptr(key), _ptr(value), _ptr(slot_mapping),
                               _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
                               _ptr(seq_lens), batch, int(max_seq_len), nb, bs, num_heads, hkv,
                               head_dim, int(sliding_window), float(scale), float(kv_scale),
                               int(num_splits), ws_ptr, ws_bytes, _stream(dev))
    _check(st, "pa_decode_fp8")
    return out


def pa_decode_num_splits(batch: int, num_heads: int, num_kv_heads: int, head_dim: int,
                         max_seq_len: int, sliding_window: int = 0, num_splits: int = 0) -> int:
    return int(load().pa_decode_num_splits(batch, num_heads, num_kv_heads, head_dim,
                                           max_seq_len, sliding_window, num_splits))


@functools.lru_cache(maxsize=1024)
def pa_decode_workspace_size(batch: int, num_heads: int, num_kv_heads: int, head_dim: int,
                             max_seq_len: int, sliding_window: int = 0,
                             num_splits: int = 0) -> int:
    return int(load().pa_decode_workspace_size(batch, num_heads, num_kv_heads, head_dim,
                                               max_seq_len, sliding_window, num_splits))


def pa_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
              block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
              scale: float, sliding_window: int = 0, num_splits: int = 0,
              key: torch.Tensor | None = None, value: torch.Tensor | None = None,
              slot_mapping: torch.Tensor | None = None, out: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Paged decode: q [B, H, D] -> out [B, H, D]; optional store of key/value first."""
    lib = load()
    dev = q.device
    _need(q, torch.bfloat16, "q", dev)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n, dev)
    _need(block_table, torch.int32, "block_table", dev)
    _need(seq_lens, torch.int32, "seq_lens", dev)
    batch, num_heads, head_dim = q.shape
    nb, bs, hkv, d = k_cache.shape
    if d != head_dim or block_table.dim() != 2 or block_table.shape[0] != batch:
        raise ValueError("pa_decode: inconsistent shapes")
    _new_tokens(key, value, slot_mapping, batch, hkv, head_dim, dev, "pa_decode")
    out = _out(out, q.shape, torch.bfloat16, dev)
    need = pa_decode_workspace_size(batch, num_heads, hkv, head_dim, max_seq_len,
                                    sliding_window, num_splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = _ptr(workspace) if need else None
    ws_bytes = workspace.numel() * workspace.element_size() if need else 0
    with _on(dev):
        st = lib.pa_decode(_ptr(out), _ptr(q), _ptr(key), _ptr(value), _ptr(slot_mapping),
                           _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
                           _ptr(seq_lens), batch, int(max_seq_len), nb, bs, num_heads, hkv,
                           head_dim, int(sliding_window), float(scale), int(num_splits), ws_ptr,
                           ws_bytes, _stream(dev))
    _check(st, "pa_decode")
    return out


def pa_decode_state_workspace_size(batch: int, num_heads: int, num_kv_heads: int,
                                   head_dim: int, max_seq_len: int, sliding_window: int = 0,
                                   num_splits: int = 0) -> int:
    return int(load().pa_decode_state_workspace_size(batch, num_heads, num_kv_heads, head_dim,
                                                     max_seq_len, sliding_window, num_splits))


def pa_decode_state(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                    block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                    scale: float, sliding_window: int = 0, num_splits: int = 0,
                    key_begin: torch.Tensor | None = None, state: torch.Tensor | None = None,
                    lse: torch.Tensor | None = None,
                    workspace: torch.Tensor | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """Partial decode over keys j >= key_begin[b]: returns (state [B, H, D] fp32,
    lse [B, H] fp32, natural log)."""
    lib = load()
    dev = q.device
    _need(q, torch.bfloat16, "q", dev)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n, dev)
    _need(block_table, torch.int32, "block_table", dev)
    _need(seq_lens, torch.int32, "seq_lens", dev)
    if key_begin is not None:
        _need(key_begin, torch.int32, "key_begin", dev)
    batch, num_heads, head_dim = q.shape
    nb, bs, hkv, d = k_cache.shape
    if d != head_dim or block_table.dim() != 2 or block_table.shape[0] != batch:
        raise ValueError("pa_decode_state: inconsistent shapes")
    state = _out(state, (batch, num_heads, head_dim), torch.float32, dev, "state")
    lse = _out(lse, (batch, num_heads), torch.float32, dev, "lse")
    need = pa_decode_state_workspace_size(batch, num_heads, hkv, head_dim, max_seq_len,
                                          sliding_window, num_splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = _ptr(workspace) if need else None
    ws_bytes = workspace.numel() * workspace.element_size() if need else 0
    with _on(dev):
        st = lib.pa_decode_state(_ptr(state), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                                 _ptr(key_begin), batch, int(max_seq_len), nb, bs, num_heads, hkv,
                                 head_dim, int(sliding_window), float(scale), int(num_splits),
                                 ws_ptr, ws_bytes, _stream(dev))
    _check(st, "pa_decode_state")
    return state, lse


def pa_merge_states(states: torch.Tensor, lses: torch.Tensor, out: torch.Tensor | None = None,
                    out_state: torch.Tensor | None = None, out_lse: torch.Tensor | None = None,
                    want_bf16: bool = True) -> torch.Tensor | None:
    """Merge partial results: states [R, ..., D] fp32, lses [R, ...] fp32 (the same rows
    in every part).  Writes any of out (bf16), out_state (fp32), out_lse; returns out."""
    lib = load()
    dev = states.device
    _need(states, torch.float32, "states", dev)
    _need(lses, torch.float32, "lses", dev)
    r = states.shape[0]
    head_dim = states.shape[-1]
    rows = states[0].numel() // head_dim
    if lses.shape[0] != r or lses[0].numel() != rows:
        raise ValueError("pa_merge_states: states and lses disagree")
    if out is not None or want_bf16:
        out = _out(out, states.shape[1:], torch.bfloat16, dev)
    if out_state is not None:
        _out(out_state, states.shape[1:], torch.float32, dev, "out_state")
    if out_lse is not None:
        _out(out_lse, lses.shape[1:], torch.float32, dev, "out_lse")
    with _on(dev):
        st = lib.pa_merge_states(_ptr(out), _ptr(out_state), _ptr(out_lse), _ptr(states),
                                 _ptr(lses), r, rows, head_dim, _stream(dev))
    _check(st, "pa_merge_states")
    return out


def pa_common_prefix_blocks(block_table, seq_lens, block_size: int) -> int:
    """Longest run of leading block-table entries shared by every request (host arrays
    or CPU tensors), limited to whole blocks inside every sequence."""
    import numpy as np
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    n = load().pa_common_prefix_blocks(bt.ctypes.data, bt.shape[0], bt.shape[1],
                                       sl.ctypes.data, int(block_size))
    if n < 0:
        raise ValueError("pa_common_prefix_blocks: invalid arguments")
    return int(n)


def pa_cascade_decode_workspace_size(batch: int, num_heads: int, num_kv_heads: int,
                                     head_dim: int, max_seq_len: int, prefix_len: int,
                                     sliding_window: int = 0) -> int:
    return int(load().pa_cascade_decode_workspace_size(batch, num_heads, num_kv_heads,
                                                       head_dim, max_seq_len, prefix_len,
                                                       sliding_window))


def pa_cascade_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                      prefix_len: int, scale: float, sliding_window: int = 0,
                      out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Decode with a prefix shared by every request (the first prefix_len / block_size
    entries of every block-table row): q [B, H, D] -> out [B, H, D]."""
    lib = load()
    dev = q.device
    _need(q, torch.bfloat16, "q", dev)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n, dev)
    _need(block_table, torch.int32, "block_table", dev)
    _need(seq_lens, torch.int32, "seq_lens", dev)
    batch, num_heads, head_dim = q.shape
    nb, bs, hkv, d = k_cache.shape
    if d != head_dim or block_table.dim() != 2 or block_table.shape[0] != batch:
        raise ValueError("pa_cascade_decode: inconsistent shapes")
    out = _out(out, q.shape, torch.bfloat16, dev)
    need = pa_cascade_decode_workspace_size(batch, num_heads, hkv, head_dim, max_seq_len,
                                            prefix_len, sliding_window)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    with _on(dev):
        st = lib.pa_cascade_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(block_table), block_table.shape[1], _ptr(seq_lens), batch,
                                   int(max_seq_len), int(prefix_len), nb, bs, num_heads, hkv,
                                   head_dim, int(sliding_window), float(scale), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(dev))
    _check(st, "pa_cascade_decode")
    return out


def pa_varlen_prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      cu_seqlens_q: torch.Tensor, seq_lens: torch.Tensor | None,
                      block_table: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int,
                      scale: float, sliding_window: int = 0,
                      cu_seqlens_k: torch.Tensor | None = None,
                      key: torch.Tensor | None = None, value: torch.Tensor | None = None,
                      slot_mapping: torch.Tensor | None = None,
                      out: torch.Tensor | None = None) -> torch.Tensor:
    """Packed varlen causal/chunked prefill: q [Tq, H, D] -> out [Tq, H, D]."""
    lib = load()
    dev = q.device
    _need(q, torch.bfloat16, "q", dev)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n, dev)
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q", dev)
    _need(block_table, torch.int32, "block_table", dev)
    if seq_lens is not None:
        _need(seq_lens, torch.int32, "seq_lens", dev)
    if cu_seqlens_k is not None:
        _need(cu_seqlens_k, torch.int32, "cu_seqlens_k", dev)
    total_q, num_heads, head_dim = q.shape
    nb, bs, hkv, d = k_cache.shape
    num_seqs = cu_seqlens_q.shape[0] - 1
    if d != head_dim or block_table.dim() != 2 or block_table.shape[0] != num_seqs:
        raise ValueError("pa_varlen_prefill: inconsistent shapes")
    _new_tokens(key, value, slot_mapping, total_q, hkv, head_dim, dev, "pa_varlen_prefill")
    out = _out(out, q.shape, torch.bfloat16, dev)
    with _on(dev):
        st = lib.pa_varlen_prefill(_ptr(out), _ptr(q), _ptr(key), _ptr(value), _ptr(slot_mapping),
                                   _ptr(k_cache), _ptr(v_cache), _ptr(cu_seqlens_q),
                                   _ptr(cu_seqlens_k), _ptr(seq_lens), _ptr(block_table),
                                   block_table.shape[1], num_seqs, total_q, int(max_seqlen_q),
                                   int(max_seqlen_k), nb, bs, num_heads, hkv, head_dim,
                                   int(sliding_window), float(scale), _stream(dev))
    _check(st, "pa_varlen_prefill")
    return out


def pa_varlen_prefill_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                          cu_seqlens_q: torch.Tensor, seq_lens: torch.Tensor | None,
                          block_table: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int,
                          scale: float, kv_scale: float, sliding_window: int = 0,
                          cu_seqlens_k: torch.Tensor | None = None,
                          key: torch.Tensor | None = None, value: torch.Tensor | None = None,
                          slot_mapping: torch.Tensor | None = None,
                          out: torch.Tensor | None = None) -> torch.Tensor:
    """pa_varlen_prefill over FP8 E4M3 caches (uint8 [NB, bs, Hkv, D], read as code *
    kv_scale); q / key / value / out bf16.  New tokens, when given, are quantised into the
    caches first."""
    lib = load()
    fn = lib.pa_varlen_prefill_fp8
    if fn.restype is not ctypes.c_int or fn.argtypes is None:
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i64,
                       i32, i32, i32, i32, i32, f32, f32, vp]
        fn.restype = ctypes.c_int
    dev = q.device
    _need(q, torch.bfloat16, "q", dev)
    _need(k_cache, torch.uint8, "k_cache", dev)
    _need(v_cache, torch.uint8, "v_cache", dev)
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q", dev)
    _need(block_table, torch.int32, "block_table", dev)
    if seq_lens is not None:
        _need(seq_lens, torch.int32, "seq_lens", dev)
    if cu_seqlens_k is not None:
        _need(cu_seqlens_k, torch.int32, "cu_seqlens_k", dev)
    total_q, num_heads, head_dim = q.shape
    nb, bs, hkv, d = k_cache.shape
    num_seqs = cu_seqlens_q.shape[0] - 1
    if (d != head_dim or v_cache.shape != k_cache.shape or block_table.dim() != 2
            or block_table.shape[0] != num_seqs):
        raise ValueError("pa_varlen_prefill_fp8: inconsistent shapes")
    _new_tokens(key, value, slot_mapping, total_q, hkv, head_dim, dev, "pa_varlen_prefill_fp8")
    out = _out(out, q.shape, torch.bfloat16, dev)
    with _on(dev):
        st = fn(_ptr(out), _ptr(q), _ptr(key), _ptr(value), _ptr(slot_mapping), _ptr(k_cache),
                _ptr(v_cache), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(seq_lens),
                _ptr(block_table), block_table.shape[1], num_seqs, total_q, int(max_seqlen_q),
                int(max_seqlen_k), nb, bs, num_heads, hkv, head_dim, int(sliding_window),
                float(scale), float(kv_scale), _stream(dev))
    _check(st, "pa_varlen_prefill_fp8")
    return out


def pa_debug_prefill_stall(stall: bool, wait_limit_ns: int = 0) -> None:
    """Testing aid: later prefill launches hand out no work item (stall) and every wait
    gives up after wait_limit_ns (0: the default 2 s), raising DEVERR_TIMEOUT."""
    lib = load()
    fn = lib.pa_debug_prefill_stall
    fn.argtypes = [ctypes.c_int, ctypes.c_uint64]
    fn.restype = ctypes.c_int
    _check(fn(1 if stall else 0, int(wait_limit_ns)), "pa_debug_prefill_stall")


def pa_read_device_error(clear: bool = True, device: torch.device | None = None) -> int:
    """Synchronise the current stream and return (and optionally clear) the device error word."""
    lib = load()
    dev = device or torch.device("cuda", torch.cuda.current_device())
    flags = ctypes.c_uint32(0)
    st = lib.pa_read_device_error(_stream(dev), ctypes.byref(flags), 1 if clear else 0)
    if st not in (PA_OK, PA_ERR_DEVICE_CHECK):
        raise PAError(st, "pa_read_device_error")
    return int(flags.value)


def pa_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                      scale: float, sliding_window: int = 0, num_splits: int = 0,
                      key: torch.Tensor | None = None, value: torch.Tensor | None = None,
                      slot_mapping: torch.Tensor | None = None,
                      out: torch.Tensor | None = None) -> torch.Tensor:
    """pa_decode without a workspace, for callers that cannot allocate device memory.

    The split-K scratch is the library's own fixed per-device array, so no workspace is
    allocated here; pass `out` to allocate nothing at all.  Calls that may overlap on
    the GPU share that array and race; see include/pa_gb300.h.
    """
    lib = load()
    fn = lib.pa_decode_noalloc
    if fn.restype is not ctypes.c_int or fn.argtypes is None:
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i64, i32, i32, i32,
                       i32, i32, f32, i32, vp]
        fn.restype = ctypes.c_int
    dev = q.device
    _need(q, torch.bfloat16, "q", dev)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n, dev)
    _need(block_table, torch.int32, "block_table", dev)
    _need(seq_lens, torch.int32, "seq_lens", dev)
    batch, num_heads, head_dim = q.shape
    nb, bs, hkv, d = k_cache.shape
    if d != head_dim or block_table.dim() != 2 or block_table.shape[0] != batch:
        raise ValueError("pa_decode_noalloc: inconsistent shapes")
    _new_tokens(key, value, slot_mapping, batch, hkv, head_dim, dev, "pa_decode_noalloc")
    out = _out(out, q.shape, torch.bfloat16, dev)
    with _on(dev):
        st = fn(_ptr(out), _ptr(q), _ptr(key), _ptr(value), _ptr(slot_mapping), _ptr(k_cache),
                _ptr(v_cache), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), batch,
                int(max_seq_len), nb, bs, num_heads, hkv, head_dim, int(sliding_window),
                float(scale), int(num_splits), _stream(dev))
    _check(st, "pa_decode_noalloc")
    return out
