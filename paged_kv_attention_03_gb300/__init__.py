"""GB300-native attention over a paged, block-structured KV cache.

The product is ``libpa_gb300.so`` (C ABI in ``include/pa_gb300.h``), built from
``csrc/`` for sm_103a.  This package is its thin Python binding (same names as the
C entry points), the build step, and the seeded input generator used by tests and
the benchmark.  Importing the package does not load the library; the first call
does, and raises if it is missing.
"""
from ._lib import (  # noqa: F401
    DEVERR_BLOCK_RANGE,
    DEVERR_QUERY_LEN,
    DEVERR_SEQ_RANGE,
    DEVERR_SEQLENS_K,
    DEVERR_SLOT_RANGE,
    DEVERR_TIMEOUT,
    DEVERR_SLOT_MISMATCH,
    EXPORTED,
    PA_ERR_CUDA,
    PA_ERR_DEVICE_CHECK,
    PA_ERR_INVALID_ARG,
    PA_ERR_UNSUPPORTED,
    PA_OK,
    PAError,
    library_path,
    load,
    pa_decode,
    pa_decode_noalloc,
    pa_decode_state,
    pa_decode_state_workspace_size,
    pa_merge_states,
    pa_cascade_decode,
    pa_cascade_decode_workspace_size,
    pa_common_prefix_blocks,
    pa_decode_fp8,
    pa_store_kvcache_fp8,
    pa_decode_num_splits,
    pa_decode_workspace_size,
    pa_read_device_error,
    pa_debug_prefill_stall,
    pa_store_kvcache,
    pa_varlen_prefill,
    pa_varlen_prefill_fp8,
    status_string,
    version,
)
from .builder import build  # noqa: F401
