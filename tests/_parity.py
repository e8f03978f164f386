"""Helpers shared by the GPU parity tests: run the oracle on host copies of a case's
inputs and compare the library's bf16 outputs with the oracle's fp64 results."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_attention_03_gb300.inputs import PagedCase, bf16_bits

# The stated bar for bf16-in / fp32-accumulate attention against the fp64 oracle.
MAX_ABS = 1e-2
MEAN_ABS = 1e-3


def host_inputs(case: PagedCase) -> dict:
    """uint16 copies of every bf16 input (taken before any kernel touches the cache)."""
    return dict(q=bf16_bits(case.q), key=bf16_bits(case.key), value=bf16_bits(case.value),
                k_cache=bf16_bits(case.k_cache), v_cache=bf16_bits(case.v_cache))


def oracle_store(case: PagedCase, h: dict) -> None:
    """Apply the step's store to the host cache copies (in place)."""
    oracle.store_kvcache(h["key"], h["value"], h["k_cache"], h["v_cache"], case.slot_mapping,
                         case.workload.block_size)


def oracle_attention(case: PagedCase, h: dict, seqs=None, window=None) -> np.ndarray:
    """Oracle output for the rows of the sequences in `seqs` (all when None), packed
    in sequence order; [rows, H, D] float64."""
    w = case.workload
    win = w.sliding_window if window is None else window
    if seqs is None:
        return oracle.paged_attention(h["q"], h["k_cache"], h["v_cache"], case.cu_seqlens_q,
                                      case.seq_lens, case.block_table, w.num_heads,
                                      w.num_kv_heads, win, w.final_scale)
    seqs = np.asarray(seqs)
    cu = case.cu_seqlens_q
    rows = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in seqs]) if len(seqs) else \
        np.zeros(0, np.int64)
    ql = case.query_lens[seqs]
    sub_cu = np.zeros(len(seqs) + 1, np.int32)
    sub_cu[1:] = np.cumsum(ql)
    return oracle.paged_attention(np.ascontiguousarray(h["q"][rows]), h["k_cache"],
                                  h["v_cache"], sub_cu, case.seq_lens[seqs],
                                  np.ascontiguousarray(case.block_table[seqs]), w.num_heads,
                                  w.num_kv_heads, win, w.final_scale)


def rows_of(case: PagedCase, seqs) -> np.ndarray:
    cu = case.cu_seqlens_q
    return np.concatenate([np.arange(cu[i], cu[i + 1]) for i in seqs])


# Significant bits of each output type: rounding a value x to it moves x by at most
# half an ulp, 2^(floor(log2|x|) - bits).
_SIG_BITS = {torch.bfloat16: 8, torch.float16: 11, torch.float32: 24}


def half_ulp(ref: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Largest change rounding |ref| to `dtype` (round to nearest) can make."""
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - _SIG_BITS[dtype]), 0.0)


def round_to(ref: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """fp64 values rounded once, to nearest even, to the significand of `dtype` (normal
    range; the exponent range of the outputs here is far from its limits)."""
    bits = _SIG_BITS[dtype]
    m, e = np.frexp(ref)                       # ref = m 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(np.ldexp(m, bits)), e - bits)  # rint: ties to even


# Parity figures of the tests that ran, printed at the end of the session.
RECORDS: list[tuple[str, dict]] = []


def assert_parity(got: torch.Tensor, ref: np.ndarray, what: str = "",
                  max_abs: float = MAX_ABS, mean_abs: float = MEAN_ABS) -> dict:
    """Two bars, both asserted:

    1. against the fp64 oracle: the stated bar is for the attention arithmetic (bf16
       operands, fp32 accumulation); the output's own rounding to its storage type adds
       up to half an ulp of the exact value, so element i may differ by
       max_abs + half_ulp(ref_i) (for |ref| < 1 at most 1e-2 + 2^-9).
    2. against the oracle rounded once to the output type: max-abs <= max_abs, except
       where that type's spacing exceeds max_abs (|ref| >= 2 for bf16), where the output
       must be the correctly rounded value or one of its two neighbours.
    The mean-abs bar is taken against the oracle rounded once to the output type: the
    rounding of the output itself (about a quarter of an ulp on average, ~1e-3 for rows of
    magnitude ~1, as a window of one key over an FP8 cache gives) is not arithmetic error.
    Both mean-abs figures are reported."""
    g = got.detach().float().cpu().double().numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    excess = err - (max_abs + half_ulp(ref, got.dtype))
    rr = round_to(ref, got.dtype)
    err_r = np.abs(g - rr)
    ulp = 2.0 * half_ulp(rr, got.dtype)
    coarse = ulp > max_abs
    stats = {"max_abs": float(err.max()) if err.size else 0.0,
             "mean_abs": float(err.mean()) if err.size else 0.0,
             "max_excess": float(excess.max()) if err.size else -max_abs,
             "max_abs_vs_rounded": float(err_r[~coarse].max()) if (~coarse).any() else 0.0,
             "mean_abs_vs_rounded": float(err_r.mean()) if err.size else 0.0,
             "coarse_elems": int(coarse.sum()),
             "elems": int(err.size)}
    RECORDS.append((what, stats))
    if err.size and stats["max_excess"] > 0:
        i = int(np.argmax(excess))
        raise AssertionError(f"{what}: |err| {err.flat[i]:.3e} at |ref| {abs(ref.flat[i]):.3f} "
                             f"exceeds {max_abs} + half an ulp ({half_ulp(ref.flat[i], got.dtype):.2e})")
    assert stats["max_abs_vs_rounded"] <= max_abs, \
        f"{what}: max-abs {stats['max_abs_vs_rounded']:.3e} against the rounded oracle > {max_abs}"
    if coarse.any():
        bad = err_r[coarse] > ulp[coarse] * 1.0000001
        assert not bad.any(), f"{what}: an output with |ref| >= 2 is more than one ulp off"
    assert stats["mean_abs_vs_rounded"] <= mean_abs, \
        f"{what}: mean-abs {stats['mean_abs_vs_rounded']:.3e} against the rounded oracle > {mean_abs}"
    return stats


def device_tensors(case: PagedCase, device) -> dict:
    """int32 metadata of the case as device tensors."""
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=device)
    return dict(cu_seqlens_q=t(case.cu_seqlens_q), seq_lens=t(case.seq_lens),
                block_table=t(case.block_table), slot_mapping=t(case.slot_mapping))
