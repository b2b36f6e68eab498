"""Partitioned mixed-precision ZeRO step on one GB300 (sm_103a).

Thin Python binding of the C ABI in ``include/zero_gb300.h``: the functions
here carry the C names and only marshal arguments (tensors or integers to
raw pointers, the current torch stream to a cudaStream_t).  Every step of
the method runs in the CUDA kernels of ``libzero_gb300.so``; there is no
CPU fallback.  The library is loaded on first use and a missing build
raises :class:`ZeroError` with the command that builds it.
"""

from ._binding import (  # noqa: F401
    ZERO_BF16, ZERO_F_DOUBLE_BUFFER, ZERO_FP16, ZERO_MAX_RANKS,
    ZERO_MODE_AUTO, ZERO_MODE_SPECULATIVE, ZERO_MODE_SPECULATIVE_STAGED, ZERO_MODE_TWO_PASS_REREAD,
    ZERO_MODE_TWO_PASS_WS, ZeroError, exported_symbols, hyper, library_path,
    load_library, zero_bytes_moved, zero_destroy, zero_gather_bucket,
    zero_get_status, zero_init_partition, zero_last_error, zero_partition_info,
    zero_reduce_scatter_bucket, zero_reduce_scatter_bucket_replicas, zero_set_scaler, zero_step,
    zero_step_noalloc, zero_noalloc_scratch_bytes, zero_quantize_blocks, zero_dequantize_blocks, zero_gather_bucket_q8,
    zero_reduce_scatter_bucket_q, ZERO_Q_BLOCK, zero_reduce_scatter_gather_bucket, zero_set_persistent,
    result_from_device, pointer_array,
)
